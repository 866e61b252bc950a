"""GPU parity: every exported call against the CPU oracle on seeded inputs.

Bit-exact: the quantized Q codes and scales. Within max|err| <= 2e-2 max|V|
and mean|err| <= 2e-3 max|V|: the bf16 output. Padding requests must stay
untouched, the device status word must stay clean.
"""

import numpy as np
import pytest

import synth
from tests._harness import SENTINEL, all_units, compare, full_workload, run_gpu, run_oracle, sample_units

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]  # MJ_IMPL_SIMT, MJ_IMPL_TCGEN05


def _skip_unsupported(impl, w):
    return None


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


def _case(name):
    if name == "ragged_hnd":
        return synth.make_case(name=name, num_seqs=6, q_len=1, h_q=32, h_k=8, page_size=16,
                               seq_lens=[1, 15, 16, 17, 300, 1000], layout="HND", pool_pages=200, seed=21)
    if name == "split_nhd":
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=32, h_k=8, page_size=64,
                               seq_lens=[5000, 9000, 300], layout="NHD", seed=22)
    if name == "spec_causal":
        return synth.make_case(name=name, num_seqs=7, q_len=4, h_q=32, h_k=8, page_size=32,
                               seq_lens=[40, 129, 700, 2000, 3, 0, 0], layout="HND", scale_mode="tensor",
                               seed=23, causal=True)
    if name == "spec_noncausal":
        return synth.make_case(name=name, num_seqs=7, q_len=4, h_q=32, h_k=8, page_size=32,
                               seq_lens=[40, 129, 700, 2000, 3, 0, 0], layout="HND", scale_mode="tensor",
                               seed=23, causal=False)
    if name == "fp6_small":
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=64, h_k=8, page_size=128,
                               seq_lens=[130, 1000, 257], layout="HND", kv_format="e2m3",
                               outlier_channels=4, seed=24)
    if name == "fp6_nhd_spec":
        return synth.make_case(name=name, num_seqs=3, q_len=2, h_q=16, h_k=4, page_size=32,
                               seq_lens=[33, 500, 1], layout="NHD", kv_format="e2m3", outlier_channels=4,
                               seed=25)
    raise KeyError(name)


SMALL = ["ragged_hnd", "split_nhd", "spec_causal", "spec_noncausal", "fp6_small", "fp6_nhd_spec"]


@pytest.mark.parametrize("name", ["tiny"] + SMALL)
def test_quantize_q_bit_exact(name):
    w = synth.tiny() if name == "tiny" else _case(name)
    got = run_gpu(w, impl=1)
    _, _, codes, desc = run_oracle(w, units=[])
    assert np.array_equal(got["q_codes"], codes)
    assert np.array_equal(got["q_descale"], desc)


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny(impl):
    w = synth.tiny()
    got = run_gpu(w, impl=impl)
    ref, lse, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), "tiny")
    np.testing.assert_allclose(got["lse"], lse, atol=2e-3, rtol=1e-4)
    assert got["status"] == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", SMALL)
def test_small_cases(impl, name):
    w = _case(name)
    _skip_unsupported(impl, w)
    got = run_gpu(w, impl=impl)
    ref, lse, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), name)
    real = w.seq_lens > 0
    np.testing.assert_allclose(got["lse"][real], lse[real], atol=2e-3, rtol=1e-4)
    assert np.all(got["lse"][~real] == SENTINEL)
    assert got["status"] == 0


@pytest.mark.parametrize("impl", IMPLS)
def test_split_equals_unsplit(impl):
    w = _case("split_nhd")
    a = run_gpu(w, impl=impl, max_splits=1)
    b = run_gpu(w, impl=impl, max_splits=16)
    assert not a["info"]["with_reduction"] and b["info"]["with_reduction"]
    assert max(b["info"]["n_splits"][: w.num_seqs]) > 1
    ref, _, _, _ = run_oracle(w)
    compare(w, a["out"], ref, all_units(w), "unsplit")
    compare(w, b["out"], ref, all_units(w), "split")
    vm = np.abs(a["out"]).max()
    assert np.abs(a["out"] - b["out"]).max() <= 2e-2 * max(vm, 1e-6)


@pytest.mark.parametrize("impl", IMPLS)
def test_upper_bound_plan_and_margin(impl):
    """Planning on longer lengths (upper bound + draft margin) must not change
    the result: masking always uses the true lengths in device memory."""
    w = _case("split_nhd")
    got = run_gpu(w, impl=impl, plan_lens=w.seq_lens + 700, margin=3)
    ref, _, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), "upper-bound plan")
    w2 = _case("ragged_hnd")
    got2 = run_gpu(w2, impl=impl, plan_lens=w2.seq_lens + 129, margin=2, ctas_per_sm=1, sm_count=20)
    ref2, _, _, _ = run_oracle(w2)
    compare(w2, got2["out"], ref2, all_units(w2), "upper-bound plan, split")


@pytest.mark.parametrize("impl", IMPLS)
def test_per_seq_descales_and_strided_output(impl):
    w = _case("ragged_hnd")
    got = run_gpu(w, impl=impl, descale_per_seq=True, out_strided=True)
    ref, _, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), "per-(seq, head) descales, strided O")


@pytest.mark.parametrize("impl", IMPLS)
def test_repeated_steps_are_identical(impl):
    w = _case("spec_causal")
    a = run_gpu(w, impl=impl, steps=1)
    b = run_gpu(w, impl=impl, steps=3)
    assert np.array_equal(a["out"], b["out"])


# ----------------------------------------------------------------------------
# the five configurations at full size, in the benchmark's launch settings
# ----------------------------------------------------------------------------
FULL = {
    "qwen3_8b_decode": dict(ctas_per_sm=2, max_splits=64, kv_stages=6),
    "long_split": dict(ctas_per_sm=4, max_splits=64),
    "long_single": dict(ctas_per_sm=2, max_splits=64),
    "spec_verify": dict(ctas_per_sm=4, max_splits=64, kv_stages=4),
    "spec_verify_noncausal": dict(ctas_per_sm=4, max_splits=64, kv_stages=4),
    "fp6_decode": dict(ctas_per_sm=2, max_splits=64, kv_stages=6),
}


# which units each full-size configuration compares with the oracle: all of
# them where the oracle finishes in seconds, else a seeded tenth plus the
# first and last request (the last is padding in spec_verify)
ALL_UNITS = {"qwen3_8b_decode", "spec_verify", "spec_verify_noncausal"}


def full_size_units(w, name, seed=3):
    if name in ALL_UNITS:
        return all_units(w)
    n = max(1, -(-w.num_seqs * w.h_k // 10))
    units = set(sample_units(w, n, seed=seed)) | {(w.num_seqs - 1, 0), (0, w.h_k - 1)}
    return sorted(units)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", list(FULL))
def test_full_size(impl, name):
    w = full_workload(name)
    _skip_unsupported(impl, w)
    got = run_gpu(w, impl=impl, **FULL[name])
    units = full_size_units(w, name)
    total = w.num_seqs * w.h_k
    assert len(units) == total if name in ALL_UNITS else 10 * len(units) >= total
    ref, lse, _, _ = run_oracle(w, units=units)
    compare(w, got["out"], ref, units, name)
    real_rows = np.repeat(w.seq_lens > 0, w.q_len)
    assert np.all(np.isfinite(got["out"][real_rows]))
    assert np.all(got["out"][~real_rows] == SENTINEL)
    for b, g in units:
        if w.seq_lens[b] > 0:
            np.testing.assert_allclose(got["lse"][b, g], lse[b, g], atol=2e-3, rtol=1e-4)
    assert got["status"] == 0


def test_tcgen05_rejects_what_it_cannot_run():
    """Packed e2m3 strides that are not multiples of 32 bytes are outside the
    packed TMA type's rules: the tensor-core variant refuses them (the
    automatic choice falls back to the CUDA-core kernel)."""
    import paged_fp8_decode_gb300 as mj

    w = synth.make_case(name="fp6_odd", num_seqs=2, q_len=1, h_q=8, h_k=1, page_size=16,
                        seq_lens=[40, 17], layout="HND", kv_format="e2m3", seed=31)
    # rows 96 B apart; insert a 16-byte gap between pages -> page stride % 32 != 0
    pool = w.k_cache.shape[0]
    for name in ("k_cache", "v_cache"):
        buf = getattr(w, name)
        wide = np.zeros((pool, buf[0].size + 16), dtype=np.uint8)
        wide[:, : buf[0].size] = buf.reshape(pool, -1)
        setattr(w, name, wide)
    w.kv_strides = (w.kv_strides[0] + 16, w.kv_strides[1], w.kv_strides[2])
    w.k_cache = w.k_cache.reshape(-1)
    w.v_cache = w.v_cache.reshape(-1)
    with pytest.raises(mj.MjError) as e:
        run_gpu(w, impl=2)
    assert e.value.status == mj.MJ_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------
# fp16 output (T5DecodeRunner's out_dtype is bf16 or fp16)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["ragged_hnd", "spec_causal", "fp6_small"])
def test_fp16_output(impl, name):
    import torch

    w = _case(name)
    got = run_gpu(w, impl=impl, out_dtype=torch.float16)
    ref, lse, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), name + " fp16")
    real = w.seq_lens > 0
    np.testing.assert_allclose(got["lse"][real], lse[real], atol=2e-3, rtol=1e-4)
    assert got["status"] == 0


@pytest.mark.parametrize("impl", IMPLS)
def test_fp16_output_split(impl):
    """The split plan: the merge kernel writes the fp16 output."""
    import torch

    w = _case("split_nhd")
    got = run_gpu(w, impl=impl, max_splits=16, out_dtype=torch.float16)
    assert got["info"]["with_reduction"]
    ref, _, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), "split fp16")
    assert got["status"] == 0


# ----------------------------------------------------------------------------
# bf16 Q as is (T5DecodeRunner's q_mode="bf16"; e4m3 KV only)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["ragged_hnd", "spec_causal", "spec_noncausal", "wide_rows"])
def test_bf16_q(impl, name):
    """The CUDA-core kernel uses Q exactly; the tensor-core kernel carries each
    value as two e4m3 terms (hi + lo, per-(request, KV head) scales)."""
    if name == "wide_rows":  # 32 query rows per (request, KV head): the widest row tile
        w = synth.make_case(name=name, num_seqs=3, q_len=4, h_q=64, h_k=8, page_size=32, seq_lens=[50, 700, 129],
                            layout="HND", scale_mode="head", seed=26)
    else:
        w = _case(name)
    got = run_gpu(w, impl=impl, q_mode="bf16")
    ref, lse, _, _ = run_oracle(w, q_mode="bf16")
    compare(w, got["out"], ref, all_units(w), name + " bf16 Q")
    real = w.seq_lens > 0
    # Two e4m3 terms carry each Q value to ~2^-8 relative (bf16's own step),
    # so the tensor-core kernel's logits, and the LSE, move by up to about
    # 2^-8 * |q| |k| * softmax_scale (~4e-3 here); the CUDA-core kernel uses Q exactly.
    np.testing.assert_allclose(got["lse"][real], lse[real], atol=1e-2 if impl == 2 else 2e-3, rtol=1e-4)
    assert got["status"] == 0, f"device status {got['status']}"


@pytest.mark.parametrize("impl", IMPLS)
def test_bf16_q_split_and_full_size(impl):
    w = _case("split_nhd")
    got = run_gpu(w, impl=impl, max_splits=16, q_mode="bf16")
    assert got["info"]["with_reduction"]
    ref, _, _, _ = run_oracle(w, q_mode="bf16")
    compare(w, got["out"], ref, all_units(w), "split bf16 Q")
    w = full_workload("qwen3_8b_decode")
    got = run_gpu(w, impl=impl, ctas_per_sm=2, max_splits=64, kv_stages=6, q_mode="bf16")
    units = sorted(set(sample_units(w, 6, seed=5)) | {(w.num_seqs - 1, w.h_k - 1)})
    ref, _, _, _ = run_oracle(w, units=units, q_mode="bf16")
    compare(w, got["out"], ref, units, "qwen3 bf16 Q")
    real_rows = np.repeat(w.seq_lens > 0, w.q_len)
    assert np.all(np.isfinite(got["out"][real_rows]))
    assert got["status"] == 0


def test_bf16_q_rejections():
    import paged_fp8_decode_gb300 as mj

    with pytest.raises(mj.MjError) as e:  # packed e2m3 KV is fp8-Q only
        run_gpu(_case("fp6_small"), impl=0, q_mode="bf16")
    assert e.value.status == mj.MJ_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------
# Q quantized inside the decode kernel (q_mode MJ_Q_FP8_FUSED): the same codes
# and descales as mj_quantize_q (which is pinned to the oracle), so the whole
# step's output is bit-identical to the step with the separate quantize call
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["ragged_hnd", "spec_causal", "fp6_small", "fp6_nhd_spec", "split", "wide_rows"])
def test_fused_quantize_is_bit_identical(impl, name):
    kw = {}
    if name == "split":
        w, kw = _case("split_nhd"), dict(max_splits=16)
    elif name == "wide_rows":  # 64 query rows per (request, KV head): two row tiles share one amax
        w = synth.make_case(name=name, num_seqs=3, q_len=8, h_q=64, h_k=8, page_size=32, seq_lens=[50, 700, 129],
                            layout="HND", scale_mode="head", seed=27)
    else:
        w = _case(name)
    a = run_gpu(w, impl=impl, **kw)
    b = run_gpu(w, impl=impl, q_mode="fp8_fused", **kw)
    assert a["status"] == 0 and b["status"] == 0
    real_rows = np.repeat(w.seq_lens > 0, w.q_len)
    assert np.array_equal(a["out"][real_rows], b["out"][real_rows])
    real = w.seq_lens > 0
    assert np.array_equal(a["lse"][real], b["lse"][real])
    assert np.all(b["out"][~real_rows] == SENTINEL)


def test_fused_quantize_full_size():
    w = full_workload("qwen3_8b_decode")
    a = run_gpu(w, impl=2, **FULL["qwen3_8b_decode"])
    b = run_gpu(w, impl=2, q_mode="fp8_fused", **FULL["qwen3_8b_decode"])
    assert np.array_equal(a["out"], b["out"]) and b["status"] == 0


def _tie_case():
    """The tiny workload with request 0's Q replaced by a hand-worked case:
    the amax element 3136 gives the descale 3136 / 448 = 7 exactly, and
    x = 12.6875 divides to exactly 1.8125, the midpoint of the e4m3 values
    1.75 (even mantissa) and 1.875. A true division rounds it to 1.75 (code
    0x3E, 0xBE for -x); a multiply by float32(1/7) would give 1.875."""
    w = synth.tiny()
    q = np.zeros_like(w.q_f32)
    q[0, 0, 0], q[0, 0, 1], q[0, 1, 5] = 3136.0, 12.6875, -12.6875
    q[w.q_len:] = w.q_f32[w.q_len:]  # request 1 keeps its ordinary values
    w.q_f32 = q.astype(np.float32)
    w.q_bits = (w.q_f32.view(np.uint32) >> 16).astype(np.uint16)  # exact: every value is a bf16 value
    return w


@pytest.mark.parametrize("impl", IMPLS)
def test_quantize_q_rounds_a_true_quotient_at_an_e4m3_tie(impl):
    w = _tie_case()
    ref, ref_lse, codes, desc = run_oracle(w)
    assert desc[0, 0] == np.float32(7.0) and codes[0, 0, 0, 1] == 0x3E and codes[0, 0, 1, 5] == 0xBE
    a = run_gpu(w, impl=impl)  # mj_quantize_q, then the decode kernel
    assert np.array_equal(a["q_codes"], codes) and np.array_equal(a["q_descale"], desc)
    compare(w, a["out"], ref, all_units(w), "e4m3 tie in Q")
    b = run_gpu(w, impl=impl, q_mode="fp8_fused")  # the decode kernel quantizes Q itself
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    assert a["status"] == 0 and b["status"] == 0
