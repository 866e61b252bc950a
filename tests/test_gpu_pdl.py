"""The decode launch may overlap the kernel before it on the stream
(programmatic dependent launch), and before it waits for that kernel its
producer warps ask L2 for the first KV tiles, aimed with the work rows and
block-table entries as they stand then. Those guesses must never reach the
result: here the kernel right before each decode rewrites the block table to
point at a second copy of the pages, after the copy the old table points at
has been overwritten with NaN codes. Every step must follow the new table
(the oracle's output, no NaN), for both bf16-input Q modes, split and not."""

import numpy as np
import pytest

import synth
from tests._harness import SENTINEL, all_units, compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


CASES = {
    "split_nhd": (dict(num_seqs=3, q_len=1, h_q=32, h_k=8, page_size=64, seq_lens=[5000, 9000, 300],
                       layout="NHD", seed=22), 16),
    "unsplit_hnd": (dict(num_seqs=80, q_len=1, h_q=32, h_k=8, page_size=16, seq_lens=[700] * 80,
                         layout="HND", seed=41), 1),
}


@pytest.mark.parametrize("q_mode", ["fp8_fused", "bf16"])
@pytest.mark.parametrize("name", list(CASES))
def test_block_table_rewritten_right_before_the_decode(name, q_mode):
    import torch

    from paged_fp8_decode_gb300 import DecodeStep, mj_workspace_status
    from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

    kw, max_splits = CASES[name]
    w = synth.make_case(name=name, **kw)
    kv = paged_kv_from_workload(w)
    P = w.num_pages
    k_orig, v_orig = kv.k_cache.clone(), kv.v_cache.clone()
    kv.k_cache = torch.cat([kv.k_cache, k_orig]).contiguous()  # copy 0: pages 0..P-1, copy 1: P..2P-1
    kv.v_cache = torch.cat([kv.v_cache, v_orig]).contiguous()
    kv.num_pages = 2 * P
    bt = [kv.block_table.clone(), torch.where(kv.block_table >= 0, kv.block_table + P, kv.block_table)]
    q = q_from_workload(w)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, max_splits=max_splits,
                      causal=w.causal, impl=2, with_lse=True, q_mode=q_mode)
    info = step.plan(w.seq_lens, w.num_seqs)
    assert bool(info["with_reduction"]) == (max_splits > 1)
    out = torch.full((w.num_seqs * w.q_len, w.h_q, w.d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ref, _, _, _ = run_oracle(w, q_mode="bf16" if q_mode == "bf16" else "fp8")
    for i in range(4):
        use = i % 2
        stale = slice(0, P) if use == 1 else slice(P, 2 * P)
        kv.k_cache[stale].fill_(0x7F)  # e4m3 NaN in the copy the new table leaves
        kv.v_cache[stale].fill_(0x7F)
        kv.block_table.copy_(bt[use])  # the last kernel before the decode
        step.run(q, out, kv, w.num_seqs, w.softmax_scale)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got)), f"step {i}: NaN from the old block table"
        compare(w, got, ref, all_units(w), f"{name} {q_mode} step {i}")
        kv.k_cache[stale].copy_(k_orig)  # restore that copy for the next step
        kv.v_cache[stale].copy_(v_orig)
    assert mj_workspace_status(step.workspace) == 0
