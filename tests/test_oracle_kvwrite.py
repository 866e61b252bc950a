"""Pins of the oracle's KV-cache write at ``slot_mapping``."""

import numpy as np
import pytest

from oracle import formats as F
from oracle import kvwrite as W

PS, NP, HK, D = 16, 6, 2, 128


def _layout(kind, kv_format):
    rb = W.row_bytes(D, kv_format)
    if kind == "HND":  # (page, head, token, row)
        return (HK * PS * rb, rb, PS * rb)
    return (PS * HK * rb, HK * rb, rb)  # NHD: (page, token, head, row)


def _pools(kv_format):
    rb = W.row_bytes(D, kv_format)
    size = NP * PS * HK * rb
    rng = np.random.default_rng(3)
    return rng.integers(0, 256, size, dtype=np.uint8), rng.integers(0, 256, size, dtype=np.uint8)


def _gather(pool, strides, slot, h, rb):
    off = (slot // PS) * strides[0] + (slot % PS) * strides[1] + h * strides[2]
    return pool[off:off + rb]


def _scales(kv_format, rng):
    if kv_format == W.KV_E4M3:
        return rng.uniform(0.002, 0.05, HK).astype(np.float32), rng.uniform(0.002, 0.05, HK).astype(np.float32)
    return rng.uniform(0.1, 2.0, (HK, D)).astype(np.float32), rng.uniform(0.1, 2.0, (HK, D)).astype(np.float32)


@pytest.mark.parametrize("kv_format", [W.KV_E4M3, W.KV_E2M3, W.KV_E3M2, W.KV_E2M1])
@pytest.mark.parametrize("kind", ["HND", "NHD"])
def test_padding_writes_nothing_and_rows_land_at_their_slots(kv_format, kind):
    rng = np.random.default_rng(11)
    T = 9
    key = rng.standard_normal((T, HK, D)).astype(np.float32)
    val = rng.standard_normal((T, HK, D)).astype(np.float32)
    slots = np.array([5, -1, 17, 40, -1, 3, 95, 64, 2], dtype=np.int64)
    ks, vs = _scales(kv_format, rng)
    kp, vp = _pools(kv_format)
    kp0, vp0 = kp.copy(), vp.copy()
    st = _layout(kind, kv_format)
    W.write_kv(key, val, kp, vp, slots, PS, st, st, kv_format, ks, vs)
    rb = W.row_bytes(D, kv_format)
    kq, vq = W.quantize_rows(key, ks, kv_format), W.quantize_rows(val, vs, kv_format)
    touched = np.zeros(kp.size, dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(HK):
            assert np.array_equal(_gather(kp, st, s, h, rb), kq[t, h])
            assert np.array_equal(_gather(vp, st, s, h, rb), vq[t, h])
            off = (s // PS) * st[0] + (s % PS) * st[1] + h * st[2]
            touched[off:off + rb] = True
    # every other byte is as it was
    assert np.array_equal(kp[~touched], kp0[~touched]) and np.array_equal(vp[~touched], vp0[~touched])


def test_e4m3_representable_rows_are_exact():
    # x = scale * v with power-of-two scales: x / scale is exactly v
    rng = np.random.default_rng(12)
    codes = rng.choice([c for c in range(256) if c not in (0x7F, 0xFF)], size=(4, HK, D)).astype(np.uint8)
    scale = np.array([2.0 ** -6, 2.0 ** 3], dtype=np.float32)
    x = (F.e4m3_decode(codes) * scale.reshape(1, HK, 1)).astype(np.float32)
    assert np.array_equal(W.quantize_rows(x, scale, W.KV_E4M3), codes)
    # per tensor: one scale for every head
    x1 = (F.e4m3_decode(codes) * np.float32(0.5)).astype(np.float32)
    assert np.array_equal(W.quantize_rows(x1, np.array([0.5], np.float32), W.KV_E4M3), codes)


def test_e2m3_representable_rows_are_exact():
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 64, size=(4, HK, D), dtype=np.uint8)
    s = (2.0 ** rng.integers(-4, 4, size=(HK, D))).astype(np.float32)
    x = (F.e2m3_decode(codes) * s).astype(np.float32)
    rows = W.quantize_rows(x, s, W.KV_E2M3)
    assert rows.shape == (4, HK, 96)
    assert np.array_equal(F.fp6_unpack_rows(rows), codes)


def test_narrow_representable_rows_are_exact():
    """Power-of-two channel scales times e3m2 / e2m1 values: x / s is exactly
    the value, so the rows hold exactly those codes."""
    rng = np.random.default_rng(16)
    s = (2.0 ** rng.integers(-4, 4, size=(HK, D))).astype(np.float32)
    for fmt, ncode, dec, unpack, rb in ((W.KV_E3M2, 64, F.e3m2_decode, F.fp6_unpack_rows, 96),
                                        (W.KV_E2M1, 16, F.e2m1_decode, F.fp4_unpack_rows, 64)):
        codes = rng.integers(0, ncode, size=(4, HK, D), dtype=np.uint8)
        x = (dec(codes) * s).astype(np.float32)
        rows = W.quantize_rows(x, s, fmt)
        assert rows.shape == (4, HK, rb) and W.row_bytes(D, fmt) == rb
        assert np.array_equal(unpack(rows), codes)


@pytest.mark.parametrize("kv_format", [W.KV_E4M3, W.KV_E2M3, W.KV_E3M2, W.KV_E2M1])
def test_rows_at_exact_midpoints_round_to_the_even_code(kv_format):
    """x / scale exactly halfway between two adjacent values of the format
    (power-of-two scales keep the quotient exact) is written as the code whose
    mantissa LSB is 0, for both signs and every adjacent pair."""
    table, n, sign, unpack = {W.KV_E4M3: (F.E4M3_TABLE, 0x7F, 0x80, None),
                              W.KV_E2M3: (F.E2M3_TABLE, 0x20, 0x20, F.fp6_unpack_rows),
                              W.KV_E3M2: (F.E3M2_TABLE, 0x20, 0x20, F.fp6_unpack_rows),
                              W.KV_E2M1: (F.E2M1_TABLE, 0x8, 0x8, F.fp4_unpack_rows)}[kv_format]
    mids = (table[: n - 1] + table[1:n]) / 2.0  # between codes i and i + 1
    want = np.array([i if i % 2 == 0 else i + 1 for i in range(n - 1)], dtype=np.uint8)
    vals = np.concatenate([mids, -mids])
    want = np.concatenate([want, want | sign])
    reps = -(-len(vals) // D)
    y = np.resize(vals, reps * HK * D).reshape(reps, HK, D)
    w = np.resize(want, reps * HK * D).reshape(reps, HK, D)
    if kv_format == W.KV_E4M3:
        scale = np.array([2.0 ** -5, 2.0 ** 2], dtype=np.float32)
        x = (y * scale.reshape(1, HK, 1)).astype(np.float32)
        codes = W.quantize_rows(x, scale, kv_format)
    else:
        scale = (2.0 ** (np.arange(HK * D).reshape(HK, D) % 7 - 3)).astype(np.float32)
        x = (y * scale).astype(np.float32)
        codes = unpack(W.quantize_rows(x, scale, kv_format))
    assert np.array_equal(x.astype(np.float64) / (scale.reshape(1, HK, 1) if kv_format == W.KV_E4M3 else scale), y)
    assert np.array_equal(codes, w)


@pytest.mark.parametrize("kv_format", [W.KV_E4M3, W.KV_E2M3, W.KV_E3M2, W.KV_E2M1])
def test_written_rows_are_within_half_a_step(kv_format):
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((64, HK, D)) * 3).astype(np.float32)
    ks, _ = _scales(kv_format, rng)
    rows = W.quantize_rows(x, ks, kv_format)
    if kv_format == W.KV_E4M3:
        codes, vals = rows, F.E4M3_TABLE[:0x7F]
        y = x / ks.reshape(1, HK, 1).astype(np.float64)
        dec = F.e4m3_decode(codes)
        top = 448.0
    else:
        unpack, table, n, top = {W.KV_E2M3: (F.fp6_unpack_rows, F.E2M3_TABLE, 0x20, 7.5),
                                 W.KV_E3M2: (F.fp6_unpack_rows, F.E3M2_TABLE, 0x20, 28.0),
                                 W.KV_E2M1: (F.fp4_unpack_rows, F.E2M1_TABLE, 0x8, 6.0)}[kv_format]
        codes, vals = unpack(rows), table[:n]
        y = x / ks.astype(np.float64)
        dec = table[codes]
    a = np.minimum(np.abs(y), top)
    i = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, len(vals) - 2)
    half_step = (vals[i + 1] - vals[i]) / 2
    # the quotient is float32: allow its own rounding (relative 2^-24)
    assert np.all(np.abs(np.abs(dec) - a) <= half_step * (1 + 1e-6) + a * 2.0 ** -23)
    assert np.all((np.signbit(dec) == np.signbit(y)) | (dec == 0))


@pytest.mark.parametrize("kv_format", [W.KV_E4M3, W.KV_E2M3, W.KV_E3M2, W.KV_E2M1])
def test_token_order_does_not_matter(kv_format):
    rng = np.random.default_rng(15)
    T = 12
    key = rng.standard_normal((T, HK, D)).astype(np.float32)
    val = rng.standard_normal((T, HK, D)).astype(np.float32)
    slots = rng.permutation(NP * PS)[:T].astype(np.int64)
    slots[3] = -1
    ks, vs = _scales(kv_format, rng)
    st = _layout("HND", kv_format)
    a_k, a_v = _pools(kv_format)
    b_k, b_v = a_k.copy(), a_v.copy()
    W.write_kv(key, val, a_k, a_v, slots, PS, st, st, kv_format, ks, vs)
    perm = rng.permutation(T)
    W.write_kv(key[perm], val[perm], b_k, b_v, slots[perm], PS, st, st, kv_format, ks, vs)
    assert np.array_equal(a_k, b_k) and np.array_equal(a_v, b_v)


@pytest.mark.parametrize("kv_format", [W.KV_E4M3, W.KV_E2M3, W.KV_E3M2, W.KV_E2M1])
def test_head_size_256_row_is_two_128_channel_rows(kv_format):
    """A 256-channel row's bytes are the two 128-channel halves' bytes side by
    side: one code per byte (e4m3), or a little-endian 6-bit (4-bit) stream
    whose first 128 codes fill exactly 96 (64) bytes. The 128-channel encoding is
    pinned by the hand-packed fixtures."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((5, HK, 256)).astype(np.float32) * 3
    if kv_format == W.KV_E4M3:
        sc = rng.uniform(0.002, 0.05, HK).astype(np.float32)
        lo, hi = sc, sc
    else:
        sc = rng.uniform(0.1, 2.0, (HK, 256)).astype(np.float32)
        lo, hi = sc[:, :128], sc[:, 128:]
    whole = W.quantize_rows(x, sc, kv_format)
    assert whole.shape == (5, HK, W.row_bytes(256, kv_format))
    halves = np.concatenate([W.quantize_rows(x[..., :128], lo, kv_format),
                             W.quantize_rows(x[..., 128:], hi, kv_format)], axis=-1)
    assert np.array_equal(whole, halves)
