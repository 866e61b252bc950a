"""Occupancy-pinned split-KV plan (oracle side).

Test infrastructure only (see :mod:`oracle`).

Sources on the ``mjolnir/runner.py`` page: ``tile_width``;
``T5DecodeRunner.n_tiles`` / ``.slots``; the capacity comment in
``T5DecodeRunner.__init__`` (grid.x is ``max(slots, max_num_seqs)``);
``T5DecodeRunner.plan`` (``lens = seq_len + margin``, the call of
``plan_split_kv(lens, h_k, n_tiles, sm_count, ctas_per_sm, max_splits,
pad_to)``, ``with_reduction = max_splits > 1 and num_seqs < slots``, a work
row ``w`` is non-empty iff ``w[2] > w[1]``). The README ("A decode step",
item 1) states the aim: exactly one wave of ``ctas_per_sm`` CTAs per SM. KV
tiles are 128 tokens (the tile length ``l2_prefetch`` names in the runner's
constructor).

The body of ``plan_split_kv`` is not on the pages. Reading (the plainest
algorithm consistent with the call site and the reduction rule):

* ``t_b = ceil((seq_len_b + margin) / 128)`` tiles per request (the margin
  is added to every request, as the page's ``plan`` does);
* without reduction: one work row per request, ``(b, 0, t_b, 0)``,
  ``chunk_tiles = max(1, max_b t_b)``, ``n_splits_b = 1``;
* with reduction: ``chunk_tiles = c``, the SMALLEST ``c >= 1`` with
  ``sum_b max(1, ceil(t_b/c)) <= slots`` and ``max_b ceil(t_b/c) <=
  max_splits``; request ``b`` gets ``n_splits_b = max(1, ceil(t_b/c))`` rows
  ``(b, s*c, min((s+1)*c, t_b), s)``, in request-major, split-minor order;
* the list is padded with ``(0, 0, 0, 0)`` rows (empty) to ``pad_to``.

Pins (``tests/test_oracle_plan.py``): ``tile_width`` against the values its
docstring fixes; exhaustive brute force over ``c`` on random small cases;
coverage of every tile exactly once; the capacity bound; ``max_splits = 1``
never splits.
"""

from __future__ import annotations

from dataclasses import dataclass

KV_TILE = 128


def tile_width(n_q: int, fp8_q: bool) -> int:
    """The query rows one CTA takes: the smallest power of two that holds
    ``n_q``, clamped to [16, 32] with fp8 Q and to [8, 32] with bf16 Q
    (``tile_width`` on the runner page)."""
    base = 16 if fp8_q else 8
    p = 1
    while p < n_q:
        p *= 2
    return max(base, min(32, p))


def n_tiles(q_len: int, h_r: int, fp8_q: bool = True) -> int:
    n_q = q_len * h_r
    tw = tile_width(n_q, fp8_q)
    return -(-n_q // tw)


def slots(sm_count: int, ctas_per_sm: int, h_k: int, n_row_tiles: int) -> int:
    return max(1, (sm_count * ctas_per_sm) // (h_k * n_row_tiles))


@dataclass
class Plan:
    work: list  # pad_to rows of [b, tile_begin, tile_end, split]
    n_splits: list  # per request
    chunk_tiles: int
    with_reduction: bool
    slots: int
    num_work: int


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def plan_split_kv(seq_lens, num_seqs: int, q_len: int, h_q: int, h_k: int, sm_count: int,
                  ctas_per_sm: int, max_splits: int, margin: int, pad_to: int,
                  fp8_q: bool = True) -> Plan:
    h_r = h_q // h_k
    nt = n_tiles(q_len, h_r, fp8_q)
    s = slots(sm_count, ctas_per_sm, h_k, nt)
    # KV tiles of each request, counted on its length grown by the margin
    t = []
    for b in range(num_seqs):
        grown = int(seq_lens[b]) + margin
        t.append(_ceil(grown, KV_TILE) if grown > 0 else 0)
    with_reduction = max_splits > 1 and num_seqs < s

    work = []
    n_splits = []
    if not with_reduction:
        chunk = max([1] + t)
        for b in range(num_seqs):
            work.append([b, 0, t[b], 0])
            n_splits.append(1)
    else:
        chunk = None
        c = 1
        while chunk is None:
            items = sum(max(1, _ceil(tb, c)) for tb in t)
            widest = max([0] + [_ceil(tb, c) for tb in t])
            if items <= s and widest <= max_splits:
                chunk = c
            c += 1
        for b in range(num_seqs):
            ns = max(1, _ceil(t[b], chunk))
            n_splits.append(ns)
            for sp in range(ns):
                work.append([b, sp * chunk, min((sp + 1) * chunk, t[b]), sp])
    if len(work) > pad_to:
        raise ValueError(f"plan needs {len(work)} work rows but pad_to is {pad_to}")
    work += [[0, 0, 0, 0] for _ in range(pad_to - len(work))]
    return Plan(work=work, n_splits=n_splits, chunk_tiles=chunk, with_reduction=with_reduction,
                slots=s, num_work=pad_to)
