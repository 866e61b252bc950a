"""Number formats of the KV cache and of quantized Q (oracle side).

Test infrastructure only (see :mod:`oracle`).

* **e4m3** (OCP FP8 E4M3, the ``float8_e4m3fn`` flavour the runner page
  uses for Q and KV; ``FP8_MAX = 448`` at the top of ``mjolnir/runner.py``):
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  is subnormal (``m/8 * 2**-6``); the all-ones pattern ``S.1111.111`` is NaN;
  there is no infinity, so the largest finite magnitude is
  ``1.75 * 2**8 = 448``.
* **e2m3** (OCP FP6 E2M3, ``kv_format="e2m3"`` in ``VariantKey`` of
  ``mjolnir/runner.py``): 1 sign bit, 2 exponent bits with bias 1, 3 mantissa
  bits; exponent field 0 is subnormal (``m/8``); no NaN and no infinity; the
  largest magnitude is ``1.875 * 2**2 = 7.5`` (the 7.5 in the fallback
  descale of ``_install_fp6_scales`` on the ``mjolnir/backend.py`` page).
* **packing**: the ``VariantKey`` comment on the runner page says e2m3 codes
  are packed "4 per 3 bytes" as a "little-endian bitstream". Reading: code
  ``i`` of a row occupies bits ``[6*i, 6*i+6)`` of the row's bytes read as one
  little-endian integer, bit 0 being the least significant bit of byte 0.
  A row of ``d`` codes is ``d*6/8`` bytes (``kv_row_bytes`` in
  ``T5DecodeRunner.__init__``).

Pins (``tests/test_oracle_formats.py``): hand-derived code values from the
format definitions (``tests/golden/e4m3_codes.txt``,
``tests/golden/e2m3_codes.txt``), exhaustive decode/encode round trips of
both formats, ties-to-even at every midpoint, saturation, agreement with
torch's own ``float8_e4m3fn`` conversion on random inputs, and hand-packed
byte fixtures (``tests/golden/fp6_packing.txt``) read in both directions.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M3_MAX = 7.5


# ----------------------------------------------------------------------------
# e4m3
# ----------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    """Value of one e4m3 code, straight from the bit fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """Codes (any integer array) -> float64 values."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# Non-negative finite e4m3 values in code order (codes 0x00..0x7E); they are
# strictly increasing, so the position of a value in this list is its code.
_E4M3_POS = E4M3_TABLE[:0x7F].copy()


def e4m3_encode(x) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to the even code, saturating.

    Plain definition: for ``|x|`` between two adjacent representable
    magnitudes ``v_i <= |x| < v_{i+1}``, pick the nearer one; at the exact
    midpoint pick the one whose mantissa LSB (= code LSB) is 0. Magnitudes
    at or above 448 give 448 (saturating, like ``cvt ... satfinite``), NaN
    gives the NaN code 0x7F, and the sign bit follows the sign of ``x``
    (so ``-0.0`` and negative values that round to zero give 0x80).
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    vals = _E4M3_POS
    i = np.searchsorted(vals, a, side="right") - 1  # vals[i] <= a
    i = np.clip(i, 0, len(vals) - 1)
    top = i >= len(vals) - 1  # a >= 448
    j = np.minimum(i + 1, len(vals) - 1)
    lo, hi = vals[i], vals[j]
    # Compare 2a with lo + hi: both sides are exact in float64 because lo and
    # hi have at most 4 significant bits and a is a float32/float64 input.
    twice = 2.0 * a
    mid = lo + hi
    up = (twice > mid) | ((twice == mid) & (i % 2 == 1))
    code = np.where(up, j, i)
    code = np.where(top, 0x7E, code).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    return code


# ----------------------------------------------------------------------------
# e2m3
# ----------------------------------------------------------------------------
def e2m3_value(code: int) -> float:
    """Value of one 6-bit e2m3 code, straight from the bit fields."""
    code = int(code) & 0x3F
    sign = -1.0 if code & 0x20 else 1.0
    e = (code >> 3) & 0x3
    m = code & 0x7
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 1)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 1)


E2M3_TABLE = np.array([e2m3_value(c) for c in range(64)], dtype=np.float64)


def e2m3_decode(codes) -> np.ndarray:
    return E2M3_TABLE[np.asarray(codes, dtype=np.uint8) & 0x3F]


# Non-negative e2m3 values in code order (codes 0x00..0x1F), strictly
# increasing: subnormals 0, 1/8 .. 7/8, then 1.0 .. 7.5.
_E2M3_POS = E2M3_TABLE[:0x20].copy()


def e2m3_encode(x) -> np.ndarray:
    """Round to the nearest e2m3 value, ties to the even code, saturating.

    The same plain definition as :func:`e4m3_encode` over the 32 non-negative
    e2m3 values: the nearer of the two neighbours, the even code (mantissa
    LSB 0) at an exact midpoint, magnitudes at or above 7.5 give 7.5 (code
    0x1F), and the sign bit (bit 5) follows the sign of ``x`` (``-0.0`` and
    negative values that round to zero give 0x20). The format has no NaN: a
    NaN input is outside the contract of the cache write.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    vals = _E2M3_POS
    i = np.searchsorted(vals, a, side="right") - 1  # vals[i] <= a
    i = np.clip(i, 0, len(vals) - 1)
    top = i >= len(vals) - 1  # a >= 7.5
    j = np.minimum(i + 1, len(vals) - 1)
    lo, hi = vals[i], vals[j]
    twice = 2.0 * a  # exact: lo, hi and a need few bits
    mid = lo + hi
    up = (twice > mid) | ((twice == mid) & (i % 2 == 1))
    code = np.where(up, j, i)
    code = np.where(top, 0x1F, code).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x20, code).astype(np.uint8)
    return code


# ----------------------------------------------------------------------------
# 4-codes-in-3-bytes little-endian bitstream
# ----------------------------------------------------------------------------
def fp6_unpack_rows(packed) -> np.ndarray:
    """Packed rows ``[..., 3*k]`` (uint8) -> codes ``[..., 4*k]`` (uint8).

    Code ``i`` of a row is bits ``[6i, 6i+6)`` of the row's little-endian
    bitstream. Written as a plain loop over codes so that it can be checked
    against the statement by eye.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    nbytes = packed.shape[-1]
    assert nbytes % 3 == 0, "a packed e2m3 row is a whole number of 3-byte groups"
    ncodes = nbytes * 8 // 6
    flat = packed.reshape(-1, nbytes).astype(np.uint32)
    out = np.zeros((flat.shape[0], ncodes), dtype=np.uint8)
    for i in range(ncodes):
        code = np.zeros(flat.shape[0], dtype=np.uint32)
        for k in range(6):
            bit = 6 * i + k
            code |= ((flat[:, bit // 8] >> (bit % 8)) & 1) << k
        out[:, i] = code
    return out.reshape(packed.shape[:-1] + (ncodes,))


def fp6_pack_rows(codes) -> np.ndarray:
    """Codes ``[..., 4*k]`` (6-bit values in uint8) -> packed rows ``[..., 3*k]``.

    The inverse of :func:`fp6_unpack_rows`: bit ``k`` of code ``i`` goes to
    bit ``6i + k`` of the row's little-endian bitstream. A plain loop over
    codes and bits.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    ncodes = codes.shape[-1]
    assert ncodes % 4 == 0, "a packed e2m3 row holds a whole number of 4-code groups"
    nbytes = ncodes * 6 // 8
    flat = codes.reshape(-1, ncodes).astype(np.uint32)
    out = np.zeros((flat.shape[0], nbytes), dtype=np.uint32)
    for i in range(ncodes):
        for k in range(6):
            bit = 6 * i + k
            out[:, bit // 8] |= ((flat[:, i] >> k) & 1) << (bit % 8)
    return out.astype(np.uint8).reshape(codes.shape[:-1] + (nbytes,))
