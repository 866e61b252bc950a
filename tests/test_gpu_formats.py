"""GPU parity of the other narrow KV formats, packed e3m2 and e2m1 (the
package README, "Beyond fp8: the harness", lists 6-bit e2m3 and e3m2 and
4-bit e2m1, all taken by tcgen05's kind::f8f6f4).

Both decode kernels against the oracle (output within max|err| <= 2e-2
max|V| and mean|err| <= 2e-3 max|V|, LSE at 2e-3), the Q quantization fused
into the decode kernel bit-identical to the separate call, split == unsplit,
and the cache write bit-exact, for each format. The tensor-core kernel reads
K in its own format (e3m2: TMA 16U6_ALIGN16B, e2m1: 16U4_ALIGN16B) and
widens V to e4m3 in shared memory.
"""

import numpy as np
import pytest

import synth
from oracle import kvwrite as OW
from tests._harness import SENTINEL, all_units, compare, run_gpu, run_oracle, sample_units

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]  # MJ_IMPL_SIMT, MJ_IMPL_TCGEN05
FORMATS = ["e3m2", "e2m1"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


def _case(name, fmt):
    if name == "gqa8_hnd":  # 8 query rows per (request, KV head), page 128
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=64, h_k=8, page_size=128,
                               seq_lens=[130, 1000, 257], layout="HND", kv_format=fmt, outlier_channels=4,
                               seed=71)
    if name == "spec_nhd":  # 2 query tokens, NHD, a 1-token request
        return synth.make_case(name=name, num_seqs=3, q_len=2, h_q=16, h_k=4, page_size=32,
                               seq_lens=[33, 500, 1], layout="NHD", kv_format=fmt, outlier_channels=4, seed=72)
    if name == "ragged_p16":  # 4 rows, page 16, ragged lengths and a padding request
        return synth.make_case(name=name, num_seqs=6, q_len=1, h_q=32, h_k=8, page_size=16,
                               seq_lens=[1, 15, 16, 17, 300, 0], layout="HND", kv_format=fmt, outlier_channels=2,
                               pool_pages=60, seed=73)
    if name == "wide_rows":  # 32 query rows (the widest row tile)
        return synth.make_case(name=name, num_seqs=2, q_len=4, h_q=64, h_k=8, page_size=64,
                               seq_lens=[90, 700], layout="HND", kv_format=fmt, outlier_channels=4, seed=74,
                               causal=False)
    if name == "split":
        return synth.make_case(name=name, num_seqs=3, q_len=1, h_q=32, h_k=8, page_size=64,
                               seq_lens=[5000, 9000, 300], layout="NHD", kv_format=fmt, outlier_channels=4, seed=75)
    raise KeyError(name)


CASES = ["gqa8_hnd", "spec_nhd", "ragged_p16", "wide_rows"]


def _check(w, got, ref, lse, label):
    compare(w, got["out"], ref, all_units(w), label)
    real = w.seq_lens > 0
    np.testing.assert_allclose(got["lse"][real], lse[real], atol=2e-3, rtol=1e-4)
    assert np.all(got["lse"][~real] == SENTINEL)
    real_rows = np.repeat(real, w.q_len)
    assert np.all(got["out"][~real_rows] == SENTINEL)
    assert got["status"] == 0, f"device status {got['status']}"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", CASES)
def test_decode(fmt, impl, name):
    w = _case(name, fmt)
    got = run_gpu(w, impl=impl)
    ref, lse, codes, desc = run_oracle(w)
    _check(w, got, ref, lse, f"{fmt} {name}")
    assert np.array_equal(got["q_codes"], codes) and np.array_equal(got["q_descale"], desc)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("impl", IMPLS)
def test_split_equals_unsplit(fmt, impl):
    w = _case("split", fmt)
    a = run_gpu(w, impl=impl, max_splits=1)
    b = run_gpu(w, impl=impl, max_splits=16)
    assert not a["info"]["with_reduction"] and b["info"]["with_reduction"]
    ref, lse, _, _ = run_oracle(w)
    _check(w, a, ref, lse, f"{fmt} unsplit")
    _check(w, b, ref, lse, f"{fmt} split")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["gqa8_hnd", "spec_nhd", "split"])
def test_fused_quantize_is_bit_identical(fmt, impl, name):
    w = _case(name, fmt)
    kw = dict(max_splits=16) if name == "split" else {}
    a = run_gpu(w, impl=impl, **kw)
    b = run_gpu(w, impl=impl, q_mode="fp8_fused", **kw)
    assert a["status"] == 0 and b["status"] == 0
    real_rows = np.repeat(w.seq_lens > 0, w.q_len)
    assert np.array_equal(a["out"][real_rows], b["out"][real_rows])


@pytest.mark.parametrize("fmt", FORMATS)
def test_bf16_q_is_refused(fmt):
    import paged_fp8_decode_gb300 as mj

    with pytest.raises(mj.MjError) as e:  # packed KV is fp8-Q only
        run_gpu(_case("gqa8_hnd", fmt), impl=0, q_mode="bf16")
    assert e.value.status == mj.MJ_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["fp6_e3m2_decode", "fp4_decode"])
def test_full_size(name):
    """The fp6 configuration's batch (128 x 8192 tokens, 64/8 heads, page 128)
    in e3m2 and e2m1, in the benchmark's launch settings: a seeded tenth of
    the (request, KV head) units plus the last one."""
    w = synth.WORKLOADS[name]()
    got = run_gpu(w, impl=0, ctas_per_sm=2, max_splits=64, kv_stages=6, q_mode="fp8_fused")
    units = sorted(set(sample_units(w, -(-w.num_seqs * w.h_k // 10), seed=3)) | {(w.num_seqs - 1, w.h_k - 1)})
    assert 10 * len(units) >= w.num_seqs * w.h_k
    ref, _, _, _ = run_oracle(w, units=units)
    compare(w, got["out"], ref, units, name)
    assert np.all(np.isfinite(got["out"]))
    assert got["status"] == 0


# ----------------------------------------------------------------------------
# the cache write
# ----------------------------------------------------------------------------
def _write(c):
    import torch

    import paged_fp8_decode_gb300 as mj

    dev = "cuda"
    key = torch.from_numpy(c.key_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    val = torch.from_numpy(c.value_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    slots = torch.from_numpy(c.slots).to(dev)
    kp = torch.from_numpy(c.k_pool.copy()).to(dev)
    vp = torch.from_numpy(c.v_pool.copy()).to(dev)
    ks = torch.from_numpy(np.ascontiguousarray(c.k_scale)).to(dev)
    vs = torch.from_numpy(np.ascontiguousarray(c.v_scale)).to(dev)
    mj.mj_write_kv(key, val, slots, kp, vp, c.kv_strides, c.page_size, c.num_pages, mj.KV_FORMATS[c.kv_format],
                   ks, vs)
    torch.cuda.synchronize()
    ok, ov = c.k_pool.copy(), c.v_pool.copy()
    fmt = {"e3m2": OW.KV_E3M2, "e2m1": OW.KV_E2M1}[c.kv_format]
    OW.write_kv(c.key, c.value, ok, ov, c.slots, c.page_size, c.kv_strides, c.kv_strides, fmt, c.k_scale,
                c.v_scale)
    return kp.cpu().numpy(), vp.cpu().numpy(), ok, ov


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("spec", [dict(num_tokens=300, num_pages=5, page_size=128, layout="HND", pad_every=9),
                                  dict(num_tokens=97, num_pages=12, page_size=16, layout="NHD", pad_every=3),
                                  dict(num_tokens=150, d=256, num_pages=4, page_size=64, layout="HND", pad_every=8)],
                         ids=["hnd", "nhd", "d256"])
def test_write_bit_exact(fmt, spec):
    c = synth.kv_write_case(name="w_" + fmt, kv_format=fmt, outlier_channels=4, seed=76, **spec)
    gk, gv, ok, ov = _write(c)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


@pytest.mark.parametrize("fmt", FORMATS)
def test_write_saturates_and_keeps_signs(fmt):
    c = synth.kv_write_case(name="sat_" + fmt, num_tokens=64, num_pages=4, page_size=16, kv_format=fmt, seed=77)
    c.k_scale = np.full_like(c.k_scale, 1e-3)  # far past the format's largest value
    c.v_scale = np.full_like(c.v_scale, 1e5)   # rounds to (signed) zero
    gk, gv, ok, ov = _write(c)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
