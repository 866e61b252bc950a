"""The allocation-free entry point, mj_decode_attention_noalloc.

It serves callers that cannot allocate device memory (an engine whose
KV-cache pool owns nearly all of HBM, a plugin under a framework's own
caching allocator): the split-KV partials live in a fixed array compiled into
the library. Checked here against the workspace-based entry points
(mj_decode_attention + mj_merge_lse) and against the CPU oracle on a
workload that really splits, on two calls in a row, within the tolerance of
the parity tests; and its status word (mj_noalloc_status) reports a page id
out of range and is cleared by the read. This file is
collected last so that a run stopping at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import synth
from tests._harness import SENTINEL, all_units, compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()
    return torch


def _setup(torch, max_splits):
    from paged_fp8_decode_gb300 import DecodeStep
    from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

    w = synth.make_case(name="noalloc_split", num_seqs=3, q_len=1, h_q=32, h_k=8, page_size=64,
                        seq_lens=[5000, 9000, 300], layout="NHD", seed=22)
    kv = paged_kv_from_workload(w)
    q = q_from_workload(w)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, ctas_per_sm=2,
                      max_splits=max_splits, causal=w.causal)
    info = step.plan(w.seq_lens, w.num_seqs)
    return w, kv, q, step, info


def test_noalloc_matches_workspace_entry_points(ready):
    torch = ready
    import paged_fp8_decode_gb300 as mj

    w, kv, q, step, info = _setup(torch, max_splits=16)
    assert info["with_reduction"] and max(info["n_splits"][: w.num_seqs]) > 1
    shape = (w.num_seqs * w.q_len, w.h_q, w.d)
    ref = torch.full(shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    step.run(q, ref, kv, w.num_seqs, w.softmax_scale)
    torch.cuda.synchronize()
    ref_np = ref.float().cpu().numpy()

    oracle_out, _, _, _ = run_oracle(w)
    lib = mj.load_library()
    stream = torch.cuda.current_stream()
    for call in range(2):
        out = torch.full(shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
        a = step.args(kv, out, w.num_seqs, w.softmax_scale)
        a.workspace, a.workspace_bytes = None, 0  # ignored by the allocation-free call
        st = lib.mj_decode_attention_noalloc(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream))
        assert st == mj.MJ_OK, lib.mj_status_string(st)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        compare(w, got, ref_np, all_units(w), f"no-alloc call {call} vs the workspace path")
        compare(w, got, oracle_out, all_units(w), f"no-alloc call {call} vs the oracle")
    assert mj.mj_noalloc_status(stream) == 0


def test_noalloc_rejects_plans_beyond_its_scratch(ready):
    torch = ready
    import paged_fp8_decode_gb300 as mj

    w, kv, q, step, info = _setup(torch, max_splits=64)
    need = mj.mj_workspace_size(step.slots, 64, w.q_len, w.h_q, w.h_k)
    assert need > mj.NOALLOC_SCRATCH_BYTES
    out = torch.full((w.num_seqs * w.q_len, w.h_q, w.d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    a = step.args(kv, out, w.num_seqs, w.softmax_scale)
    with pytest.raises(mj.MjError) as e:
        mj.mj_decode_attention_noalloc(a)
    assert e.value.status == mj.MJ_ERR_CAPACITY
    torch.cuda.synchronize()
    assert np.all(out.float().cpu().numpy() == SENTINEL)  # nothing was enqueued


def test_noalloc_status_reports_a_bad_page(ready):
    """A block-table entry past the pool: the CUDA-core kernel skips that
    page and records it in the scratch's status word, which
    mj_noalloc_status reads (bit 1) and clears."""
    torch = ready
    import paged_fp8_decode_gb300 as mj

    w, kv, q, step, info = _setup(torch, max_splits=16)
    stream = torch.cuda.current_stream()
    assert mj.mj_noalloc_status(stream) == 0
    kv.block_table[0, 3] = w.num_pages + 5
    out = torch.full((w.num_seqs * w.q_len, w.h_q, w.d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    mj.mj_quantize_q(q, w.num_seqs, w.q_len, w.h_k, step.q_codes, step.q_descale, stream=stream)
    a = step.args(kv, out, w.num_seqs, w.softmax_scale)
    a.impl = mj.MJ_IMPL_SIMT
    mj.mj_decode_attention_noalloc(a, stream)
    assert mj.mj_noalloc_status(stream) & 1
    assert mj.mj_noalloc_status(stream) == 0  # the read cleared it
