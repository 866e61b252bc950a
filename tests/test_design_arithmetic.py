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
  max(2^-8 p, 2^-10) of p (pair A).
* P as the kernel carries it, pair A and, where p < 1/4, pair B (the same
  split of what pair A left, times 2^10, weighed 2^-10), is within
  max(2^-8 p, 2^-20) of p, so keys down to 27 binades below the reference
  max keep their weight; on a long row with one dominant key that keeps the
  output within tolerance of exact softmax, where pair A alone does not.
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


def _e4(x):
    return F.e4m3_decode(F.e4m3_encode(np.asarray(x, dtype=np.float32)))


def _pair(x):
    """hi + lo: x as two e4m3 terms (float32 arithmetic, as in the kernel)."""
    x = np.asarray(x, dtype=np.float32)
    hi = _e4(x)
    return hi + _e4((x - hi.astype(np.float32)).astype(np.float32))


def _kernel_p(p):
    """p as the tensor-core kernel carries it: pair A, hi = e4m3(p) and
    lo = e4m3(p - hi); where p < 1/4 also pair B, the same split of
    (p - hi - lo) * 2^10 (exact in float32), weighed 2^-10."""
    p = np.asarray(p, dtype=np.float32)
    hi = _e4(p)
    d = (p - hi.astype(np.float32)).astype(np.float32)
    lo = _e4(d)
    y = np.where(p < np.float32(0.25), ((d - lo.astype(np.float32)) * np.float32(1024.0)).astype(np.float32),
                 np.float32(0.0))
    return hi + lo + _pair(y) / 1024.0


def test_p_as_four_e4m3_terms():
    p = (2.0 ** np.linspace(-40.0, 8.6, 400001)).astype(np.float32).astype(np.float64)
    err = np.abs(_kernel_p(p) - p)
    assert np.all(err <= np.maximum(2.0 ** -8 * p, 2.0 ** -20))
    keep = p >= 2.0 ** -8  # full relative precision down to 16 binades below the max
    assert np.all(err[keep] <= 2.0 ** -8 * p[keep])
    # pair B never saturates: below 1/4, p * 2^10 < 256 < 448
    assert _e4(np.float32(0.25 * 1024.0 * (1 - 2.0 ** -24))) < 448.0


def test_range_of_p():
    """Pair A alone keeps every key down to 17 binades below the reference
    max (p = 2^-9, e4m3's smallest subnormal) and loses every key 18 or more
    binades below it (p = 2^-10 ties between 0 and 2^-9 and rounds to the
    even code, 0). With pair B the same holds 10 binades further down: keys
    to 27 binades below the max keep their weight exactly."""
    for gap in range(0, 18):
        assert _pair(2.0 ** (8 - gap)) == 2.0 ** (8 - gap)
    for gap in range(18, 30):
        assert _pair(2.0 ** (8 - gap)) == 0.0
    for gap in range(0, 28):
        assert _kernel_p(2.0 ** (8 - gap)) == 2.0 ** (8 - gap)
    for gap in range(28, 40):
        assert _kernel_p(2.0 ** (8 - gap)) == 0.0


@pytest.mark.parametrize("n", [32768, 131072])
def test_dominant_key_over_a_long_row(n):
    """One key 20 binades above n near-equal others (an attention sink over
    a long row): the kernel's P arithmetic against exact softmax. With pair
    A alone the others round to zero and the output is the sink's V; their
    true share, n * 2^-20 of the sink's weight, is then lost."""
    rng = np.random.default_rng(7)
    t = rng.standard_normal(n) * 0.05  # log2 units; the others near 0
    t[0] = 20.0
    v = 1.0 + 0.25 * rng.standard_normal((n, 8))
    v[0] = -2.0
    vmax = np.abs(v).max()
    p = 2.0 ** (t - t.max())
    exact = (p[:, None] * v).sum(0) / p.sum()
    pk = (2.0 ** (t - t.max() + 8)).astype(np.float32)

    def out(w, l):
        return (w[:, None] * v).sum(0) / l.sum()

    a = _pair(pk)
    err_a = np.abs(out(a, a) - exact).max() / vmax  # l from the represented weights
    err_k = np.abs(out(_kernel_p(pk), pk) - exact).max() / vmax  # the kernel: l sums the p themselves
    assert err_a > 2e-2, "the case must lie beyond pair A's reach"
    assert err_k < 2e-3, f"four terms: {err_k:.2e} of max|V|"
