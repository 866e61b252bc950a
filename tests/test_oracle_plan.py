"""Pins of the oracle's split-KV plan."""

import itertools

import numpy as np
import pytest

from oracle import plan as P


def test_tile_width_values():
    # next power of two >= n_q, floor 16 (fp8 Q) / 8 (bf16 Q), cap 32
    assert [P.tile_width(n, True) for n in (1, 4, 8, 16, 17, 32, 33, 64)] == [16, 16, 16, 16, 32, 32, 32, 32]
    assert [P.tile_width(n, False) for n in (1, 4, 8, 9, 16, 31, 32, 100)] == [8, 8, 8, 16, 16, 32, 32, 32]


def test_n_tiles_and_slots():
    assert P.n_tiles(1, 4) == 1 and P.n_tiles(4, 4) == 1 and P.n_tiles(1, 8) == 1
    assert P.n_tiles(3, 16) == 2  # 48 rows in 32-row tiles
    assert P.slots(20, 2, 8, 1) == 5  # the pages' Thor: one wave of 2 x 20 CTAs over 8 heads
    assert P.slots(152, 2, 8, 1) == 38
    assert P.slots(10, 1, 64, 1) == 1  # never below one
    # more query rows than one 32-row tile: the slots are shared by the row tiles
    assert P.slots(152, 2, 8, 2) == 19 and P.slots(152, 2, 8, 3) == 12
    p = P.plan_split_kv([4096] * 18, 18, 8, 64, 8, 152, 2, 16, 0, 64)  # 8 x 8 = 64 rows: 2 tiles
    assert P.n_tiles(8, 8) == 2 and p.slots == 19 and p.with_reduction  # 18 requests < 19 slots
    p = P.plan_split_kv([4096] * 19, 19, 8, 64, 8, 152, 2, 16, 0, 64)
    assert p.slots == 19 and not p.with_reduction


def _check_plan(p, lens, margin, num_seqs, pad_to, max_splits, slots):
    t = [-(-(L + margin) // 128) if L + margin > 0 else 0 for L in lens[:num_seqs]]
    assert len(p.work) == pad_to
    covered = {b: [] for b in range(num_seqs)}
    for b, a, e, s in p.work:
        if e > a:
            covered[b].append((s, a, e))
    for b in range(num_seqs):
        segs = sorted(covered[b])
        tiles = [x for _, a, e in segs for x in range(a, e)]
        assert tiles == list(range(t[b])), (b, segs)  # every tile once, splits in order
        assert p.n_splits[b] >= max(1, len(segs))
        assert all(e - a <= p.chunk_tiles for _, a, e in segs)
    if p.with_reduction:
        assert sum(p.n_splits) <= slots
        assert max([0] + p.n_splits) <= max_splits
    else:
        assert all(n == 1 for n in p.n_splits)


def _brute_chunk(t, slots, max_splits):
    for c in itertools.count(1):
        ok = sum(max(1, -(-x // c)) for x in t) <= slots and max([0] + [-(-x // c) for x in t]) <= max_splits
        if ok:
            return c


@pytest.mark.parametrize("seed", range(40))
def test_random_plans_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    num_seqs = int(rng.integers(0, 12))
    lens = [int(x) for x in rng.integers(0, 5000, size=num_seqs)]
    if num_seqs and rng.random() < 0.3:
        lens[-1] = 0  # trailing padding request
    h_k = int(rng.choice([1, 2, 8]))
    h_q = h_k * int(rng.choice([1, 4, 8]))
    q_len = int(rng.integers(1, 5))
    sm, cps = int(rng.choice([20, 152])), int(rng.integers(1, 5))
    max_splits = int(rng.choice([1, 2, 16, 64]))
    margin = int(rng.integers(0, 4))
    s = P.slots(sm, cps, h_k, P.n_tiles(q_len, h_q // h_k))
    pad_to = max(s, num_seqs)
    p = P.plan_split_kv(lens, num_seqs, q_len, h_q, h_k, sm, cps, max_splits, margin, pad_to)
    assert p.slots == s
    assert p.with_reduction == (max_splits > 1 and num_seqs < s)
    _check_plan(p, lens, margin, num_seqs, pad_to, max_splits, s)
    if p.with_reduction:
        t = [-(-(L + margin) // 128) if L + margin > 0 else 0 for L in lens]
        assert p.chunk_tiles == _brute_chunk(t, s, max_splits)


def test_max_splits_one_never_splits():
    p = P.plan_split_kv([131072], 1, 1, 32, 8, 152, 2, 1, 0, 38)
    assert not p.with_reduction and p.n_splits == [1]
    assert p.work[0] == [0, 0, 1024, 0]


def test_single_long_sequence_fills_one_wave():
    # 1 x 131072 tokens, 8 KV heads, 152 SMs x 2: 38 slots; max_splits >= slots
    p = P.plan_split_kv([131072], 1, 1, 32, 8, 152, 2, 64, 0, 38)
    assert p.with_reduction and p.n_splits == [38] and p.chunk_tiles == 27
    assert sum(1 for w in p.work if w[2] > w[1]) == 38


def test_full_batch_does_not_split():
    p = P.plan_split_kv([4096] * 64, 64, 1, 32, 8, 152, 2, 16, 0, 64)
    assert not p.with_reduction and p.chunk_tiles == 32
    assert p.work[:2] == [[0, 0, 32, 0], [1, 0, 32, 0]]


def test_pad_to_too_small_raises():
    with pytest.raises(ValueError):
        P.plan_split_kv([100] * 10, 10, 1, 32, 8, 152, 2, 16, 0, 5)


def test_margin_extends_plan():
    p0 = P.plan_split_kv([128], 1, 1, 8, 8, 1, 1, 1, 0, 1)
    p1 = P.plan_split_kv([128], 1, 1, 8, 8, 1, 1, 1, 1, 1)
    assert p0.work[0] == [0, 0, 1, 0] and p1.work[0] == [0, 0, 2, 0]
