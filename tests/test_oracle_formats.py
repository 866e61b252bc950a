"""Pins of the oracle's number formats (e4m3, e2m3, e3m2, e2m1, fp6 and fp4 packing)."""

import math

import numpy as np
import torch

from oracle import formats as F


def _parse_value(s):
    return float("nan") if s == "nan" else float(s)


def test_e4m3_golden_values(golden):
    for row in golden("e4m3_codes.txt"):
        code_s, val_s = row.split()[:2]
        code, want = int(code_s, 16), _parse_value(val_s)
        got = F.e4m3_value(code)
        if math.isnan(want):
            assert math.isnan(got), code_s
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code_s


def test_e2m3_golden_values(golden):
    for row in golden("e2m3_codes.txt"):
        code_s, val_s = row.split()[:2]
        code, want = int(code_s, 16), _parse_value(val_s)
        got = F.e2m3_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code_s


def test_e4m3_table_shape_and_order():
    t = F.E4M3_TABLE
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.sum(np.isnan(t)) == 2
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)  # strictly increasing with the code
    assert np.array_equal(t[0x80:0xFF], -pos)  # sign symmetry
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    back = F.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_e4m3_midpoints_go_to_even():
    pos = F.E4M3_TABLE[:0x7F]
    for c in range(0x7E):
        mid = (pos[c] + pos[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert F.e4m3_encode(mid) == even, hex(c)
        assert F.e4m3_encode(-mid) == (even | 0x80), hex(c)
        # just off the midpoint goes to the nearer neighbour
        eps = (pos[c + 1] - pos[c]) * 1e-6
        assert F.e4m3_encode(mid - eps) == c
        assert F.e4m3_encode(mid + eps) == c + 1


def test_e4m3_saturation_and_nan():
    assert F.e4m3_encode(448.0) == 0x7E
    assert F.e4m3_encode(460.0) == 0x7E
    assert F.e4m3_encode(1e9) == 0x7E
    assert F.e4m3_encode(-1e9) == 0xFE
    assert F.e4m3_encode(float("nan")) == 0x7F
    assert F.e4m3_encode(-0.0) == 0x80
    assert F.e4m3_encode(0.0) == 0x00
    assert F.e4m3_encode(2.0 ** -11) == 0x00  # below half the smallest subnormal
    assert F.e4m3_encode(2.0 ** -10) == 0x00  # exact half: tie to even (0)
    assert F.e4m3_encode(3 * 2.0 ** -11) == 0x01  # 0.75 * 2^-9 rounds up to 2^-9


def test_e4m3_matches_torch_conversion():
    """torch's float8_e4m3fn conversion is round-to-nearest-even; on the
    range the Q path produces (|x| <= 448) it must agree bit for bit."""
    rng = np.random.default_rng(7)
    xs = [
        rng.uniform(-448, 448, 200000),
        rng.standard_normal(200000) * 3,
        rng.uniform(-0.05, 0.05, 200000),  # subnormal neighbourhood
        np.ldexp(rng.uniform(1, 2, 50000), rng.integers(-12, 9, 50000)) * rng.choice([-1, 1], 50000),
    ]
    x = np.concatenate(xs).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = F.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e2m3_every_value_is_an_e4m3_value():
    """Each e2m3 value is exactly representable in e4m3 (2 exponent bits and
    3 mantissa bits fit inside 4 and 3): a property of the two formats."""
    for c in range(64):
        v = F.e2m3_value(c)
        code = F.e4m3_encode(v)
        assert F.e4m3_value(int(code)) == v


def test_e2m3_range():
    t = F.E2M3_TABLE
    assert t.max() == 7.5 and t.min() == -7.5
    assert np.all(np.diff(t[:32]) > 0)
    assert np.array_equal(t[32:], -t[:32])


def test_fp6_unpack_golden(golden):
    for row in golden("fp6_packing.txt"):
        codes_s, bytes_s = row.split("|")
        codes = [int(x) for x in codes_s.split()]
        raw = np.array([int(x, 16) for x in bytes_s.split()], dtype=np.uint8)
        got = F.fp6_unpack_rows(raw[None, :])[0]
        assert list(got) == codes, row


def test_fp6_unpack_matches_independent_packer():
    """The synthetic cache writer packs with shifts; the oracle unpacks bit
    by bit: two independent statements of the same bitstream reading."""
    from synth import pack_e2m3

    rng = np.random.default_rng(3)
    codes = rng.integers(0, 64, size=(50, 128)).astype(np.uint8)
    packed = pack_e2m3(codes)
    assert packed.shape == (50, 96)
    assert np.array_equal(F.fp6_unpack_rows(packed), codes)


# ----------------------------------------------------------------------------
# e2m3 encoder (the cache write) and the packing direction of the fixtures
# ----------------------------------------------------------------------------
def test_e2m3_roundtrip_all_codes():
    codes = np.arange(64, dtype=np.uint8)
    assert np.array_equal(F.e2m3_encode(F.e2m3_decode(codes)), codes)


def test_e2m3_midpoints_go_to_even():
    pos = F.E2M3_TABLE[:0x20]
    assert np.all(np.diff(pos) > 0)
    for c in range(0x1F):
        mid = (pos[c] + pos[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert F.e2m3_encode(mid) == even, hex(c)
        assert F.e2m3_encode(-mid) == (even | 0x20), hex(c)
        eps = (pos[c + 1] - pos[c]) * 1e-6
        assert F.e2m3_encode(mid - eps) == c
        assert F.e2m3_encode(mid + eps) == c + 1


def test_e2m3_hand_values():
    # worked by hand from the value list of tests/golden/e2m3_codes.txt
    cases = [
        (0.0625, 0x00),   # tie 0 | 0.125 -> even code 0
        (0.1875, 0x02),   # tie 0.125 (1) | 0.25 (2) -> 2
        (0.9375, 0x08),   # tie 0.875 (7) | 1.0 (8) -> 8: rounds up into the normals
        (1.0625, 0x08),   # tie 1.0 (8) | 1.125 (9) -> 8
        (1.9375, 0x10),   # tie 1.875 (15) | 2.0 (16) -> 16
        (5.5, 0x1B),      # exact: 1.375 * 4
        (5.75, 0x1C),     # tie 5.5 (27) | 6.0 (28) -> 28
        (7.4, 0x1F),      # nearer to 7.5 than to 7.0
        (7.5, 0x1F), (8.0, 0x1F), (1e30, 0x1F),  # saturation
        (-3.0, 0x34), (-0.0, 0x20), (-0.01, 0x20),
    ]
    for x, want in cases:
        assert F.e2m3_encode(x) == want, (x, hex(int(F.e2m3_encode(x))))


def test_fp6_pack_golden(golden):
    for row in golden("fp6_packing.txt"):
        codes_s, bytes_s = row.split("|")
        codes = np.array([int(v) for v in codes_s.split()], dtype=np.uint8)
        want = np.array([int(v, 16) for v in bytes_s.split()], dtype=np.uint8)
        assert np.array_equal(F.fp6_pack_rows(codes), want), row


def test_fp6_pack_unpack_inverse():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 64, size=(7, 128), dtype=np.uint8)
    packed = F.fp6_pack_rows(codes)
    assert packed.shape == (7, 96)
    assert np.array_equal(F.fp6_unpack_rows(packed), codes)


# ----------------------------------------------------------------------------
# e3m2 and e2m1 (the other narrow KV formats) and the fp4 packing
# ----------------------------------------------------------------------------
def test_e3m2_golden_values(golden):
    for row in golden("e3m2_codes.txt"):
        code_s, val_s = row.split()[:2]
        code, want = int(code_s, 16), _parse_value(val_s)
        got = F.e3m2_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code_s


def test_e2m1_golden_values(golden):
    rows = golden("e2m1_codes.txt")
    assert len(rows) == 16  # every code
    for row in rows:
        code_s, val_s = row.split()[:2]
        code, want = int(code_s, 16), _parse_value(val_s)
        got = F.e2m1_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code_s


def test_narrow_tables_order_and_range():
    for t, n, top in ((F.E3M2_TABLE, 32, 28.0), (F.E2M1_TABLE, 8, 6.0)):
        assert np.all(np.diff(t[:n]) > 0)
        assert np.array_equal(t[n:], -t[:n])
        assert t.max() == top and t.min() == -top


def test_narrow_roundtrip_all_codes():
    c6 = np.arange(64, dtype=np.uint8)
    assert np.array_equal(F.e3m2_encode(F.e3m2_decode(c6)), c6)
    c4 = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.e2m1_encode(F.e2m1_decode(c4)), c4)


def test_narrow_midpoints_go_to_even():
    for enc, pos, sign in ((F.e3m2_encode, F.E3M2_TABLE[:0x20], 0x20), (F.e2m1_encode, F.E2M1_TABLE[:0x8], 0x8)):
        for c in range(len(pos) - 1):
            mid = (pos[c] + pos[c + 1]) / 2
            even = c if c % 2 == 0 else c + 1
            assert enc(mid) == even, hex(c)
            assert enc(-mid) == (even | sign), hex(c)
            eps = (pos[c + 1] - pos[c]) * 1e-6
            assert enc(mid - eps) == c and enc(mid + eps) == c + 1


def test_narrow_hand_values():
    # worked by hand from the value lists of the e3m2 / e2m1 fixtures
    e3m2 = [(0.03125, 0x00), (0.09375, 0x02), (0.21875, 0x04), (0.28125, 0x04), (9.0, 0x18),
            (26.0, 0x1E), (27.0, 0x1F), (28.0, 0x1F), (30.0, 0x1F), (1e30, 0x1F), (-1.0, 0x2C), (-0.0, 0x20)]
    for x, want in e3m2:
        assert F.e3m2_encode(x) == want, (x, hex(int(F.e3m2_encode(x))))
    e2m1 = [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
            (5.1, 0x7), (6.0, 0x7), (100.0, 0x7), (-0.0, 0x8), (-3.0, 0xD), (-0.2, 0x8)]
    for x, want in e2m1:
        assert F.e2m1_encode(x) == want, (x, hex(int(F.e2m1_encode(x))))


def test_narrow_values_are_e4m3_values():
    """Every e3m2 and e2m1 value is exactly an e4m3 value (fewer exponent and
    mantissa bits, a range inside e4m3's): a property of the formats."""
    for value in [F.e3m2_value(c) for c in range(64)] + [F.e2m1_value(c) for c in range(16)]:
        assert F.e4m3_value(int(F.e4m3_encode(value))) == value


def test_fp4_golden(golden):
    for row in golden("fp4_packing.txt"):
        codes_s, bytes_s = row.split("|")
        codes = np.array([int(v) for v in codes_s.split()], dtype=np.uint8)
        raw = np.array([int(v, 16) for v in bytes_s.split()], dtype=np.uint8)
        assert np.array_equal(F.fp4_pack_rows(codes), raw), row
        assert np.array_equal(F.fp4_unpack_rows(raw), codes), row


def test_fp4_matches_independent_packer():
    from synth import pack_e2m1

    rng = np.random.default_rng(4)
    codes = rng.integers(0, 16, size=(40, 128)).astype(np.uint8)
    packed = pack_e2m1(codes)
    assert packed.shape == (40, 64)
    assert np.array_equal(F.fp4_unpack_rows(packed), codes)
    assert np.array_equal(F.fp4_pack_rows(codes), packed)


def test_narrow_encoders_match_independent_writer():
    """The synthetic cache writer encodes e3m2 through torch's e5m2
    conversion and e2m1 by per-binade rint; the oracle searches the value
    table. Both must give the same codes, ties and saturation included."""
    import synth

    rng = np.random.default_rng(9)
    t3, t1 = F.E3M2_TABLE[:0x20], F.E2M1_TABLE[:0x8]
    mids3 = (t3[:-1] + t3[1:]) / 2
    mids1 = (t1[:-1] + t1[1:]) / 2
    for enc, ref, table, mids, top in ((F.e3m2_encode, synth._e3m2_codes, t3, mids3, 28.0),
                                       (F.e2m1_encode, synth._e2m1_codes, t1, mids1, 6.0)):
        x = np.concatenate([rng.uniform(-1.2 * top, 1.2 * top, 100000), rng.standard_normal(100000),
                            rng.uniform(-0.3, 0.3, 50000), table, -table, mids, -mids, [0.0, -0.0, 1e9, -1e9]])
        x = x.astype(np.float32)
        assert np.array_equal(enc(x), ref(x))
