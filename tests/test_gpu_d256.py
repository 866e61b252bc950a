"""GPU parity at head size 256 (T5DecodeRunner accepts any head_size that is a
multiple of 128; the kernels are built for 128 and 256).

Same bars as at 128: Q codes and scales bit-exact, the output within
max|err| <= 2e-2 max|V| and mean|err| <= 2e-3 max|V| of the oracle, padding
rows untouched, the device status clean. Each row tile the kernels have is
covered: 4, 8, 16 and 32 query rows per (request, KV head). The tensor-core
kernel reads a 256-byte row as two 128-byte sub-tiles; the CUDA-core kernel
takes 32-row tiles as two 16-row halves. Packed e2m3 at 256 runs on the
CUDA-core kernel only.
"""

import numpy as np
import pytest

import synth
from tests._harness import SENTINEL, all_units, compare, full_workload, run_gpu, run_oracle, sample_units

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]  # MJ_IMPL_SIMT, MJ_IMPL_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


def _case(name):
    if name == "rows4_ragged":  # n_q = 4
        return synth.make_case(name=name, num_seqs=6, q_len=1, h_q=16, h_k=4, d=256, page_size=16,
                               seq_lens=[1, 15, 16, 17, 300, 1000], layout="HND", pool_pages=120, seed=61)
    if name == "rows8_split_nhd":  # n_q = 8, long enough to split
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=32, h_k=4, d=256, page_size=64,
                               seq_lens=[5000, 9000, 300], layout="NHD", seed=62)
    if name == "rows16_spec":  # n_q = 16, causal, padding requests
        return synth.make_case(name=name, num_seqs=7, q_len=4, h_q=16, h_k=4, d=256, page_size=32,
                               seq_lens=[40, 129, 700, 2000, 3, 0, 0], layout="HND", scale_mode="tensor",
                               seed=63, causal=True)
    if name == "rows32_wide":  # n_q = 32
        return synth.make_case(name=name, num_seqs=3, q_len=4, h_q=64, h_k=8, d=256, page_size=32,
                               seq_lens=[50, 700, 129], layout="HND", scale_mode="head", seed=64, causal=False)
    if name == "fp6":
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=32, h_k=4, d=256, page_size=64,
                               seq_lens=[130, 1000, 257], layout="HND", kv_format="e2m3", outlier_channels=4,
                               seed=65)
    raise KeyError(name)


E4M3 = ["rows4_ragged", "rows8_split_nhd", "rows16_spec", "rows32_wide"]


def _check(w, got, ref, lse, label, lse_atol=2e-3):
    compare(w, got["out"], ref, all_units(w), label)
    real = w.seq_lens > 0
    np.testing.assert_allclose(got["lse"][real], lse[real], atol=lse_atol, rtol=1e-4)
    assert np.all(got["lse"][~real] == SENTINEL)
    real_rows = np.repeat(real, w.q_len)
    assert np.all(got["out"][~real_rows] == SENTINEL)
    assert got["status"] == 0, f"device status {got['status']}"


@pytest.mark.parametrize("name", E4M3 + ["fp6"])
def test_quantize_q_bit_exact(name):
    w = _case(name)
    got = run_gpu(w, impl=1)
    _, _, codes, desc = run_oracle(w, units=[])
    assert np.array_equal(got["q_codes"], codes)
    assert np.array_equal(got["q_descale"], desc)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", E4M3)
def test_e4m3(impl, name):
    w = _case(name)
    got = run_gpu(w, impl=impl)
    ref, lse, _, _ = run_oracle(w)
    _check(w, got, ref, lse, name)


def test_e2m3_runs_on_cuda_cores():
    import paged_fp8_decode_gb300 as mj

    w = _case("fp6")
    ref, lse, _, _ = run_oracle(w)
    for impl in (0, 1):  # automatic choice and the CUDA-core kernel
        got = run_gpu(w, impl=impl)
        _check(w, got, ref, lse, f"fp6 impl {impl}")
    with pytest.raises(mj.MjError) as e:  # the tensor-core kernel takes packed e2m3 at D = 128 only
        run_gpu(w, impl=2)
    assert e.value.status == mj.MJ_ERR_UNSUPPORTED


@pytest.mark.parametrize("impl", IMPLS)
def test_split_equals_unsplit(impl):
    w = _case("rows8_split_nhd")
    a = run_gpu(w, impl=impl, max_splits=1)
    b = run_gpu(w, impl=impl, max_splits=16)
    assert not a["info"]["with_reduction"] and b["info"]["with_reduction"]
    assert max(b["info"]["n_splits"][: w.num_seqs]) > 1
    ref, lse, _, _ = run_oracle(w)
    _check(w, a, ref, lse, "unsplit")
    _check(w, b, ref, lse, "split (merge at D = 256)")


@pytest.mark.parametrize("kv_stages,ctas_per_sm", [(2, 2), (4, 1), (6, 1)])
def test_ring_depths(kv_stages, ctas_per_sm):
    """The tensor-core kernel's ring of 32 KB entries at several depths (the
    default 2 keeps two CTAs per SM; deeper rings take one)."""
    w = _case("rows16_spec")
    got = run_gpu(w, impl=2, kv_stages=kv_stages, ctas_per_sm=ctas_per_sm)
    ref, lse, _, _ = run_oracle(w)
    _check(w, got, ref, lse, f"stages {kv_stages}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["rows4_ragged", "rows16_spec", "rows32_wide"])
def test_bf16_q(impl, name):
    w = _case(name)
    got = run_gpu(w, impl=impl, q_mode="bf16")
    ref, lse, _, _ = run_oracle(w, q_mode="bf16")
    # the tensor-core kernel carries Q as two e4m3 terms (about 2^-8 relative)
    _check(w, got, ref, lse, name + " bf16 Q", lse_atol=1e-2 if impl == 2 else 2e-3)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["rows4_ragged", "rows16_spec", "rows32_wide", "split", "fp6"])
def test_fused_quantize_is_bit_identical(impl, name):
    kw = {}
    if name == "split":
        w, kw = _case("rows8_split_nhd"), dict(max_splits=16)
    else:
        w = _case(name)
    if name == "fp6" and impl == 2:
        pytest.skip("packed e2m3 at D = 256 runs on the CUDA-core kernel")
    a = run_gpu(w, impl=impl, **kw)
    b = run_gpu(w, impl=impl, q_mode="fp8_fused", **kw)
    assert a["status"] == 0 and b["status"] == 0
    real_rows = np.repeat(w.seq_lens > 0, w.q_len)
    assert np.array_equal(a["out"][real_rows], b["out"][real_rows])
    real = w.seq_lens > 0
    assert np.array_equal(a["lse"][real], b["lse"][real])
    assert np.all(b["out"][~real_rows] == SENTINEL)


@pytest.mark.parametrize("impl", IMPLS)
def test_fp16_output_split(impl):
    import torch

    w = _case("rows8_split_nhd")
    got = run_gpu(w, impl=impl, max_splits=16, out_dtype=torch.float16)
    assert got["info"]["with_reduction"]
    ref, lse, _, _ = run_oracle(w)
    _check(w, got, ref, lse, "split fp16")


@pytest.mark.parametrize("impl", IMPLS)
def test_full_size(impl):
    """The 64 x 4096-token batch at head size 256, in the benchmark's launch
    settings (fused Q quantization): a seeded tenth of the (request, KV head)
    units plus the first and the last."""
    w = full_workload("d256_decode")
    got = run_gpu(w, impl=impl, ctas_per_sm=2, max_splits=64, q_mode="fp8_fused")
    units = sorted(set(sample_units(w, -(-w.num_seqs * w.h_k // 10), seed=3)) | {(w.num_seqs - 1, w.h_k - 1),
                                                                                  (0, 0)})
    assert 10 * len(units) >= w.num_seqs * w.h_k
    ref, _, _, _ = run_oracle(w, units=units)
    compare(w, got["out"], ref, units, "d256_decode")
    assert np.all(np.isfinite(got["out"]))
    assert got["status"] == 0
