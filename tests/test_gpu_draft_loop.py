"""A fused multi-step draft decode: one plan, several steps, one CUDA graph.

The mjolnir/backend.py page (MjolnirMetadataBuilder.__init__) describes the
speculative drafter's loop: one set of draft metadata serves all of the
drafter's steps, and the device sequence lengths grow in place from step to
step. So the plan is made with num_speculative_tokens of headroom
(``margin``), and the kernel masks with the current device lengths.

Here each of K draft steps writes its new token's K/V rows into the cache
(mj_write_kv), advances the device lengths by one, and runs quantize, decode
and merge. All K steps are captured in one CUDA graph on a plan made once
with margin K, and the graph is replayed. Every step's output is checked
against the oracle: the oracle's own cache write of the same rows, then
attention at that step's lengths.
"""

import copy

import numpy as np
import pytest

import synth
from oracle import kvwrite as OW
from tests._harness import compare, run_oracle

pytestmark = pytest.mark.gpu

K = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


@pytest.mark.parametrize("q_mode", ["fp8", "fp8_fused"])
@pytest.mark.parametrize("ctas_per_sm,max_splits", [(2, 1), (8, 16)], ids=["unsplit", "split"])
def test_draft_steps_in_one_graph(ctas_per_sm, max_splits, q_mode):
    """q_mode fp8: cache write, length advance, mj_quantize_q, decode, merge;
    fp8_fused: the decode kernel quantizes Q and follows the length advance
    directly, so it must see that kernel's write."""
    import torch

    import paged_fp8_decode_gb300 as mj
    from paged_fp8_decode_gb300 import DecodeStep
    from paged_fp8_decode_gb300.step import paged_kv_from_workload

    base = np.array([40, 129, 300, 1000, 17, 255], dtype=np.int32)  # lengths before the draft steps
    # the cache is laid out for the final lengths (its pages exist); the first
    # lengths are what the device sees at the start
    w = synth.make_case(name="draft", num_seqs=len(base), q_len=1, h_q=32, h_k=8, page_size=16,
                        seq_lens=base + K, layout="HND", scale_mode="head", seed=51)
    B, hk, d, ps = w.num_seqs, w.h_k, w.d, w.page_size
    rng = np.random.default_rng(52)

    def bf16(x):
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)

    # per step: the draft token's Q, and its K/V rows with their slots
    q_steps = [bf16(rng.standard_normal((B, w.h_q, d))) for _ in range(K)]
    kv_new = [bf16(rng.standard_normal((2, B, hk, d))) for _ in range(K)]
    slots = []
    for s in range(K):
        pos = base + s
        slots.append(np.array([w.block_table[b, pos[b] // ps] * ps + pos[b] % ps for b in range(B)], np.int64))

    dev = "cuda"
    kv = paged_kv_from_workload(w, dev)
    kv.seq_lens.copy_(torch.from_numpy(base))
    step = DecodeStep(max_num_seqs=B, q_len=1, h_q=w.h_q, h_k=hk, d=d, ctas_per_sm=ctas_per_sm,
                      max_splits=max_splits, margin=K, causal=w.causal, impl=mj.MJ_IMPL_AUTO, q_mode=q_mode)
    step.plan(base, B)  # once, with K tokens of headroom
    torch.cuda.synchronize()
    q_dev = [q.to(dev) for q in q_steps]
    kv_dev = [t.to(dev) for t in kv_new]
    slot_dev = [torch.from_numpy(s_).to(dev) for s_ in slots]
    outs = [torch.zeros(B, w.h_q, d, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    args = [step.args(kv, outs[s], B, w.softmax_scale, q=q_dev[s] if q_mode == "fp8_fused" else None)
            for s in range(K)]

    def draft_steps():
        for s in range(K):
            mj.mj_write_kv(kv_dev[s][0], kv_dev[s][1], slot_dev[s], kv.k_cache, kv.v_cache, kv.k_strides, ps,
                           w.num_pages, mj.MJ_KV_E4M3, kv.k_descale, kv.v_descale, scale_per_head=True)
            kv.seq_lens.add_(1)
            step.run(q_dev[s], outs[s], kv, B, w.softmax_scale, args=args[s])

    # one eager decode before capture (first-call set-up such as kernel
    # attributes happens outside the graph); its output is overwritten below
    step.run(q_dev[0], outs[0], kv, B, w.softmax_scale, args=args[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        draft_steps()
    g.replay()
    torch.cuda.synchronize()
    assert mj.mj_workspace_status(step.workspace) == 0
    assert np.array_equal(kv.seq_lens.cpu().numpy(), base + K)

    # the oracle, step by step
    ow = copy.deepcopy(w)
    assert ow.k_cache.flags["C_CONTIGUOUS"] and ow.v_cache.flags["C_CONTIGUOUS"]  # reshape(-1) is a view
    for s in range(K):
        kvf = kv_new[s].float().numpy()
        OW.write_kv(kvf[0], kvf[1], ow.k_cache.reshape(-1), ow.v_cache.reshape(-1), slots[s], ps, ow.kv_strides,
                    ow.kv_strides, OW.KV_E4M3, ow.k_scale, ow.v_scale)
        ow.seq_lens = (base + s + 1).astype(np.int32)
        ow.q_f32 = q_steps[s].float().numpy().reshape(B, w.h_q, d)
        ref, _, _, _ = run_oracle(ow)
        units = [(b, g_) for b in range(B) for g_ in range(hk)]
        compare(ow, outs[s].float().cpu().numpy(), ref, units, f"draft step {s}")
