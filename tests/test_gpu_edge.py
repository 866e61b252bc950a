"""Edge cases of the decode step on the GPU: batches with little or nothing to attend.

* Every request is padding (seq_len 0, the trailing requests a serving
  engine pads a batch with): no output row and no LSE may be written, and
  the device status word stays clean, with and without split-KV reduction,
  for e4m3 and for packed e2m3.
* An empty batch (num_seqs 0) on buffers sized for a larger one: every call
  returns MJ_OK and touches nothing.
* Causal blocks as long as their request (q_len == seq_len: row t sees keys
  0..t) and longer (rows that see no key at all write 0), against the oracle.
"""

import numpy as np
import pytest

import synth
from tests._harness import SENTINEL, all_units, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]  # MJ_IMPL_SIMT, MJ_IMPL_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


def _all_padding(kv_format):
    if kv_format == "fp8":
        return synth.make_case(name="all_padding", num_seqs=5, q_len=2, h_q=32, h_k=8, page_size=16,
                               seq_lens=[0] * 5, layout="HND", seed=41)
    return synth.make_case(name="all_padding_e2m3", num_seqs=3, q_len=1, h_q=64, h_k=8, page_size=128,
                           seq_lens=[0] * 3, layout="HND", kv_format="e2m3", outlier_channels=4, seed=42)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("kv_format", ["fp8", "e2m3"])
@pytest.mark.parametrize("max_splits", [1, 16])
@pytest.mark.parametrize("q_mode", ["fp8", "fp8_fused"])
def test_all_padding_batch_writes_nothing(impl, kv_format, max_splits, q_mode):
    w = _all_padding(kv_format)
    got = run_gpu(w, impl=impl, max_splits=max_splits, q_mode=q_mode)
    assert bool(got["info"]["with_reduction"]) == (max_splits > 1)
    assert np.all(got["out"] == SENTINEL)
    assert np.all(got["lse"] == SENTINEL)
    assert got["status"] == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("q_mode", ["fp8", "fp8_fused", "bf16"])
def test_empty_batch_is_a_no_op(impl, q_mode):
    import torch

    from paged_fp8_decode_gb300 import DecodeStep, mj_workspace_status
    from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

    w = synth.make_case(name="empty_batch", num_seqs=2, q_len=1, h_q=32, h_k=8, page_size=16,
                        seq_lens=[40, 300], layout="HND", seed=43)
    kv = paged_kv_from_workload(w)
    q = q_from_workload(w)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, impl=impl,
                      max_splits=16, causal=w.causal, with_lse=True, q_mode=q_mode)
    info = step.plan(np.zeros(0, dtype=np.int32), 0)
    assert info["num_seqs"] == 0
    out = torch.full((w.num_seqs * w.q_len, w.h_q, w.d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    step.lse.fill_(SENTINEL)
    step.run(q, out, kv, 0, w.softmax_scale)
    torch.cuda.synchronize()
    assert torch.all(out == SENTINEL).item()
    assert torch.all(step.lse == SENTINEL).item()
    assert mj_workspace_status(step.workspace) == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("max_splits", [1, 16])
def test_causal_block_as_long_as_or_longer_than_its_request(impl, max_splits):
    # seq_len 4 with q_len 4: row t sees keys 0..t. seq_len 1 and 2: the first
    # rows see no key at all (written as 0). 129: one key past a tile edge.
    w = synth.make_case(name="causal_short", num_seqs=5, q_len=4, h_q=32, h_k=8, page_size=16,
                        seq_lens=[4, 1, 2, 129, 0], layout="HND", scale_mode="tensor", seed=44, causal=True)
    got = run_gpu(w, impl=impl, max_splits=max_splits)
    ref, ref_lse, _, _ = run_oracle(w)
    compare(w, got["out"], ref, all_units(w), "short causal blocks")
    real = w.seq_lens > 0
    np.testing.assert_allclose(got["lse"][real], ref_lse[real], atol=2e-3, rtol=1e-4)
    assert np.all(got["lse"][~real] == SENTINEL)
    # the first three rows of request 1 see no key: exactly 0, LSE -inf
    assert np.all(got["out"][1 * w.q_len:1 * w.q_len + 3] == 0.0)
    assert np.all(np.isneginf(got["lse"][1][:, : 3 * w.h_r]))
    assert got["status"] == 0
