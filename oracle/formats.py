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
* **packing**: the ``VariantKey`` comment on the runner page packs four e2m3
  codes into every three bytes and reads them as a little-endian stream of
  bits. Reading: code
  ``i`` of a row occupies bits ``[6*i, 6*i+6)`` of the row's bytes read as one
  little-endian integer, bit 0 being the least significant bit of byte 0.
  A row of ``d`` codes is ``d*6/8`` bytes (``kv_row_bytes`` in
  ``T5DecodeRunner.__init__``).

* **e3m2** (OCP FP6 E3M2) and **e2m1** (OCP FP4 E2M1): the other narrow KV
  formats the package README lists in "Beyond fp8: the harness" (6-bit
  ``e2m3`` and ``e3m2``, 4-bit ``e2m1``; tcgen05's ``kind::f8f6f4`` takes all
  three). The
  pages name them only; the codecs are the OCP definitions. e3m2: 1 sign
  bit, 3 exponent bits with bias 3, 2 mantissa bits, subnormals ``m/4 *
  2**-2``, largest ``1.75 * 2**4 = 28``. e2m1: 1 sign bit, 2 exponent bits
  with bias 1, 1 mantissa bit, subnormal ``m/2``, largest ``1.5 * 2**2 = 6``.
  Neither has NaN or infinity.
* **packing** of those (readings): e3m2 rows as e2m3 rows (both are fp6);
  e2m1 rows as a little-endian bitstream of 4-bit codes, code ``i`` at bits
  ``[4*i, 4*i+4)`` (low nibble first), ``d/2`` bytes per row.

Pins (``tests/test_oracle_formats.py``): hand-derived code values from the
format definitions (``tests/golden/e4m3_codes.txt``,
``tests/golden/e2m3_codes.txt``, ``tests/golden/e3m2_codes.txt``,
``tests/golden/e2m1_codes.txt``), exhaustive decode/encode round trips of
every format, ties-to-even at every midpoint, saturation, agreement with
torch's own ``float8_e4m3fn`` conversion on random inputs, and hand-packed
byte fixtures (``tests/golden/fp6_packing.txt``,
``tests/golden/fp4_packing.txt``) read in both directions.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M3_MAX = 7.5
E3M2_MAX = 28.0
E2M1_MAX = 6.0


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
# e3m2 and e2m1
# ----------------------------------------------------------------------------
def e3m2_value(code: int) -> float:
    """Value of one 6-bit e3m2 code, straight from the bit fields."""
    code = int(code) & 0x3F
    sign = -1.0 if code & 0x20 else 1.0
    e = (code >> 2) & 0x7
    m = code & 0x3
    if e == 0:
        return sign * (m / 4.0) * 2.0 ** (1 - 3)
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 3)


def e2m1_value(code: int) -> float:
    """Value of one 4-bit e2m1 code, straight from the bit fields."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * (m / 2.0) * 2.0 ** (1 - 1)
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E3M2_TABLE = np.array([e3m2_value(c) for c in range(64)], dtype=np.float64)
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e3m2_decode(codes) -> np.ndarray:
    return E3M2_TABLE[np.asarray(codes, dtype=np.uint8) & 0x3F]


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def _nearest_code(x, pos_values, sign_bit: int) -> np.ndarray:
    """The plain rounding rule of :func:`e2m3_encode` over a format's
    non-negative values in code order (strictly increasing): the nearer
    neighbour, the even code at an exact midpoint, saturation at the largest
    magnitude, and the sign bit set when ``x`` has its sign bit set."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    vals = pos_values
    n = len(vals)
    i = np.searchsorted(vals, a, side="right") - 1  # vals[i] <= a
    i = np.clip(i, 0, n - 1)
    top = i >= n - 1
    j = np.minimum(i + 1, n - 1)
    twice = 2.0 * a  # exact: the values need few bits
    mid = vals[i] + vals[j]
    up = (twice > mid) | ((twice == mid) & (i % 2 == 1))
    code = np.where(up, j, i)
    code = np.where(top, n - 1, code).astype(np.uint8)
    return np.where(np.signbit(x), code | sign_bit, code).astype(np.uint8)


def e3m2_encode(x) -> np.ndarray:
    """Round to the nearest e3m2 value, ties to the even code, saturating at
    28 (code 0x1F); sign bit 5 follows the sign of ``x``. NaN is outside the
    contract (the format has none)."""
    return _nearest_code(x, E3M2_TABLE[:0x20], 0x20)


def e2m1_encode(x) -> np.ndarray:
    """Round to the nearest e2m1 value, ties to the even code, saturating at 6
    (code 0x7); sign bit 3 follows the sign of ``x``. NaN is outside the
    contract."""
    return _nearest_code(x, E2M1_TABLE[:0x8], 0x8)


# ----------------------------------------------------------------------------
# 2-codes-per-byte little-endian bitstream (e2m1 rows)
# ----------------------------------------------------------------------------
def fp4_unpack_rows(packed) -> np.ndarray:
    """Packed rows ``[..., k]`` (uint8) -> codes ``[..., 2*k]``: code ``i`` is
    bits ``[4i, 4i+4)`` of the row's little-endian bitstream (a plain loop)."""
    packed = np.asarray(packed, dtype=np.uint8)
    nbytes = packed.shape[-1]
    flat = packed.reshape(-1, nbytes).astype(np.uint32)
    out = np.zeros((flat.shape[0], 2 * nbytes), dtype=np.uint8)
    for i in range(2 * nbytes):
        code = np.zeros(flat.shape[0], dtype=np.uint32)
        for k in range(4):
            bit = 4 * i + k
            code |= ((flat[:, bit // 8] >> (bit % 8)) & 1) << k
        out[:, i] = code
    return out.reshape(packed.shape[:-1] + (2 * nbytes,))


def fp4_pack_rows(codes) -> np.ndarray:
    """Codes ``[..., 2*k]`` (4-bit values in uint8) -> packed rows ``[..., k]``;
    the inverse of :func:`fp4_unpack_rows` (bit ``k`` of code ``i`` to bit
    ``4i + k``)."""
    codes = np.asarray(codes, dtype=np.uint8)
    ncodes = codes.shape[-1]
    assert ncodes % 2 == 0, "a packed e2m1 row holds a whole number of bytes"
    flat = codes.reshape(-1, ncodes).astype(np.uint32)
    out = np.zeros((flat.shape[0], ncodes // 2), dtype=np.uint32)
    for i in range(ncodes):
        for k in range(4):
            bit = 4 * i + k
            out[:, bit // 8] |= ((flat[:, i] >> k) & 1) << (bit % 8)
    return out.astype(np.uint8).reshape(codes.shape[:-1] + (ncodes // 2,))


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
