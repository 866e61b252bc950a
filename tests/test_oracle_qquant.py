"""Pins of the oracle's dynamic per-(request, KV head) e4m3 Q quantization."""

import numpy as np
import torch

from oracle import formats as F
from oracle.qquant import quantize_q

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
FINITE_VALS = F.e4m3_decode(FINITE)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _case(seed=0, B=3, ql=2, h_q=8, h_k=2, d=128):
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal((B * ql, h_q, d)) * rng.uniform(0.1, 5)), B, ql, h_q, h_k, d


def test_amax_element_maps_to_448():
    q, B, ql, h_q, h_k, d = _case()
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    vals = F.e4m3_decode(codes)
    for b in range(B):
        for g in range(h_k):
            assert np.abs(vals[b, g]).max() == 448.0


def test_constant_q_gives_0x7e():
    B, ql, h_q, h_k, d = 2, 1, 4, 1, 128
    q = np.full((B * ql, h_q, d), 0.75, np.float32)
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    assert np.all(codes == 0x7E)
    assert np.all(scale == np.float32(0.75) / np.float32(448))


def test_zero_q_uses_the_floor():
    B, ql, h_q, h_k, d = 1, 1, 4, 2, 128
    q = np.zeros((1, h_q, d), np.float32)
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    assert np.all(codes == 0)
    assert np.all(scale == np.float32(np.float32(1e-6) / np.float32(448)))


def test_scale_is_correctly_rounded_quotient():
    q, B, ql, h_q, h_k, d = _case(1)
    _, scale = quantize_q(q, B, ql, h_q, h_k, d)
    x = q.reshape(B, ql, h_k, h_q // h_k, d)
    amax = np.abs(x).max(axis=(1, 3, 4)).astype(np.float64)
    want = (amax / 448.0).astype(np.float32)  # float64 quotient rounded once to float32
    assert np.array_equal(scale, want)


def test_codes_use_a_true_division_not_a_reciprocal_multiply():
    """Hand-worked case where x / scale and x * (1/scale) round apart.

    The amax element 3136 gives scale = 3136 / 448 = 7 exactly. For
    x = 12.6875 the IEEE float32 quotient is exactly 1.8125, the midpoint of
    the e4m3 values 1.75 (mantissa 6, even) and 1.875, so ties-to-even gives
    1.75 (code 0x3E; 0xBE for -x). float32(1/7) is 1/7 * (1 + 4.5e-8), and
    12.6875 * float32(1/7) rounds to 1.8125 + 2^-23, which would give 1.875.
    All three inputs are exact in bf16."""
    B, ql, h_q, h_k, d = 1, 1, 2, 1, 128
    q = np.zeros((1, h_q, d), np.float32)
    q[0, 0, 0] = 3136.0
    q[0, 0, 1] = 12.6875
    q[0, 1, 5] = -12.6875
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    assert scale[0, 0] == np.float32(7.0)
    assert codes[0, 0, 0, 0] == 0x7E
    assert codes[0, 0, 0, 1] == 0x3E
    assert codes[0, 0, 1, 5] == 0xBE


def test_every_code_is_the_nearest_e4m3_value():
    """Independent of the encoder: search all finite codes for the nearest
    value to x/scale and break ties towards the even code."""
    q, B, ql, h_q, h_k, d = _case(2, B=2, ql=1, h_q=4, h_k=1, d=128)
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    x = q.reshape(B, ql, h_k, h_q // h_k, d)
    y = (x / scale[:, None, :, None, None]).astype(np.float32).astype(np.float64)
    y = y.transpose(0, 2, 1, 3, 4).reshape(B, h_k, -1, d)
    dist = np.abs(y[..., None] - FINITE_VALS)  # [..., 254]
    best = dist.min(axis=-1)
    got = np.abs(y - F.e4m3_decode(codes))
    assert np.array_equal(got, best)
    ties = (dist == best[..., None]).sum(axis=-1) > 1
    assert np.all((codes[ties] & 1) == 0)


def test_q_mul_applies_before_amax():
    B, ql, h_q, h_k, d = 1, 1, 4, 1, 128
    q = np.ones((1, h_q, d), np.float32)
    q_mul = np.ones((h_q, d), np.float32)
    q_mul[2, 5] = 4.0
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d, q_mul=q_mul)
    assert scale[0, 0] == np.float32(4.0) / np.float32(448)
    assert codes[0, 0, 2, 5] == 0x7E
    assert F.e4m3_value(int(codes[0, 0, 0, 0])) == 112.0  # 448/4


def test_row_order_is_token_major_then_gqa_head():
    """Packed row t*h_r + r holds query token t of query head g*h_r + r."""
    B, ql, h_q, h_k, d = 1, 3, 8, 2, 128
    h_r = h_q // h_k
    q = np.zeros((B * ql, h_q, d), np.float32)
    for t in range(ql):
        for h in range(h_q):
            q[t, h, :] = 1.0 + t * 16 + h  # all distinct, exact in bf16
    codes, scale = quantize_q(q, B, ql, h_q, h_k, d)
    for g in range(h_k):
        for t in range(ql):
            for r in range(h_r):
                v = F.e4m3_value(int(codes[0, g, t * h_r + r, 0])) * float(scale[0, g])
                want = 1.0 + t * 16 + g * h_r + r
                assert abs(v - want) <= want * 2 ** -4
