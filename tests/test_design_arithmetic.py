"""The arithmetic the tensor-core decode kernel is built on, checked on the CPU
with the oracle's codecs. These are properties of the number formats that the
kernel's design relies on; the GPU parity tests check the kernel itself.

* V widening: a packed code becomes an e4m3 code by moving bits, and the
  e4m3 value is the packed value times a fixed power of two (2^-6 for e2m3
  and e2m1, 2^-4 for e3m2), for every code. The kernel folds that power of
  two into the V descale.
* P = 2^(t - m_ref + 8) with t <= m_ref + 0.6 (the rescale threshold) stays
  below e4m3's largest value, so the hi term never saturates.
* P as two e4m3 terms, hi = e4m3(p) and lo = e4m3(p - hi), is within
  max(2^-8 p, 2^-10) of p.
* bf16 Q as two e4m3 terms with per-unit scales amax/448 and
  max|residual|/448 is within amax/28^2 of q: each term's rounding error is at
  most half a step of e4m3's top binade, 16/448 = 1/28 of its scale.
"""

import numpy as np
import pytest

from oracle import formats as F


def _sign_to_bit7(code: int, sign_bit: int) -> int:
    return 0x80 if code & sign_bit else 0


@pytest.mark.parametrize("fmt,ncodes,value,widen,factor", [
    # e2m3: the 5 magnitude bits keep their place
    ("e2m3", 64, F.e2m3_value, lambda c: (c & 0x1F) | _sign_to_bit7(c, 0x20), 2.0 ** -6),
    # e3m2: the 5 magnitude bits move up one place
    ("e3m2", 64, F.e3m2_value, lambda c: ((c & 0x1F) << 1) | _sign_to_bit7(c, 0x20), 2.0 ** -4),
    # e2m1: the 3 magnitude bits move up two places
    ("e2m1", 16, F.e2m1_value, lambda c: ((c & 0x7) << 2) | _sign_to_bit7(c, 0x8), 2.0 ** -6),
])
def test_v_widening_is_an_exact_bit_move(fmt, ncodes, value, widen, factor):
    for c in range(ncodes):
        e4 = widen(c)
        assert e4 & 0x7F != 0x7F, f"{fmt} code {c:#x} would widen to the e4m3 NaN code"
        assert F.e4m3_value(e4) == value(c) * factor, f"{fmt} code {c:#x}"


def test_p_below_the_rescale_threshold_never_saturates():
    tau = 0.6
    p_max = 2.0 ** (8 + tau)
    assert p_max < 448.0
    hi = F.e4m3_decode(F.e4m3_encode(np.float32(p_max)))
    assert hi < 448.0 and abs(hi - p_max) <= p_max * 2.0 ** -4


def test_p_as_two_e4m3_terms():
    p = (2.0 ** np.linspace(-20.0, 8.6, 200001)).astype(np.float32).astype(np.float64)
    hi = F.e4m3_decode(F.e4m3_encode(p))
    lo = F.e4m3_decode(F.e4m3_encode((p - hi).astype(np.float32)))
    err = np.abs(hi + lo - p)
    assert np.all(err <= np.maximum(2.0 ** -8 * p, 2.0 ** -10))
    assert np.all(err[p >= 1.0] <= 2.0 ** -8 * p[p >= 1.0])


def test_bf16_q_as_two_e4m3_terms():
    rng = np.random.default_rng(0)
    for trial in range(200):
        q = (rng.standard_normal(512) * rng.uniform(0.01, 100.0)).astype(np.float32)
        if trial % 4 == 0:
            q[rng.integers(0, 512, 4)] *= 30.0  # a few outliers
        amax = np.float32(np.abs(q).max())
        s_hi = np.float32(amax / np.float32(448.0))
        hi = F.e4m3_decode(F.e4m3_encode((q / s_hi).astype(np.float32)))
        res = (q - (hi * s_hi).astype(np.float32)).astype(np.float32)
        rmax = np.float32(np.abs(res).max())
        assert rmax <= amax / 28.0 * (1 + 2.0 ** -20)
        s_lo = np.float32(rmax / np.float32(448.0)) if rmax > 0 else np.float32(1.0)
        lo = F.e4m3_decode(F.e4m3_encode((res / s_lo).astype(np.float32)))
        err = np.abs(hi * s_hi + lo * s_lo - q)
        assert err.max() <= amax / 784.0 * (1 + 2.0 ** -16)


def test_range_of_p_in_two_e4m3_terms():
    """P = 2^(t - m_ref + 8) in two e4m3 terms keeps every key down to 17
    binades below the reference max (p = 2^-9, e4m3's smallest subnormal)
    and loses every key 18 or more binades below it (p = 2^-10 is a tie
    between 0 and 2^-9 and rounds to the even code, 0). So a row of N keys
    loses at most a share N * 2^-18 of the top key's weight, a limit of the
    representation that long rows with one dominant key can reach."""
    def two_terms(p):
        hi = F.e4m3_decode(F.e4m3_encode(np.float32(p)))
        return hi + F.e4m3_decode(F.e4m3_encode(np.float32(p - hi)))

    for gap in range(0, 18):
        p = 2.0 ** (8 - gap)
        assert two_terms(p) == p
    for gap in range(18, 30):
        assert two_terms(2.0 ** (8 - gap)) == 0.0
    # one key 18 binades above N others: the others' whole share is lost
    n = 131072
    lost = n * 2.0 ** -18 / (1 + n * 2.0 ** -18)
    assert abs(lost - 1 / 3) < 1e-12
