"""Shared test plumbing: run a synthetic workload through the C ABI on the
GPU, or through the CPU oracle, and compare them. The two sides share only
the seeded workload (synth); neither imports the other."""

from __future__ import annotations

import numpy as np

from oracle import attention as OA
from oracle.qquant import quantize_q as oracle_quantize_q

SENTINEL = -12288.0  # exact in bf16 and fp16 (-1.5 * 2^13); a padding row that still holds it was not written
ATOL_MAX = 2e-2  # max |err| <= 2e-2 * max|V|
ATOL_MEAN = 2e-3  # mean |err| <= 2e-3 * max|V|


_last_workload = {}


def full_workload(name):
    """synth.WORKLOADS[name](), kept while consecutive tests use the same
    one (a full-size batch takes seconds to generate and GBs to hold)."""
    import synth

    if name not in _last_workload:
        _last_workload.clear()
        _last_workload[name] = synth.WORKLOADS[name]()
    return _last_workload[name]


def run_gpu(w, *, impl=0, ctas_per_sm=2, max_splits=16, margin=0, plan_lens=None, sm_count=None,
            kv_stages=0, out_strided=False, descale_per_seq=False, steps=1, out_dtype=None, q_mode="fp8"):
    import torch

    from paged_fp8_decode_gb300 import DecodeStep, mj_workspace_status
    from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

    kv = paged_kv_from_workload(w)
    if descale_per_seq:  # expand to (B, h_k) with the same values
        def expand(t):
            full = t.reshape(-1).expand(w.h_k) if t.numel() == 1 else t
            return full.reshape(1, w.h_k).repeat(w.num_seqs, 1).contiguous()
        kv.k_descale, kv.v_descale = expand(kv.k_descale), expand(kv.v_descale)
        kv.descale_strides = (w.h_k, 1)
    q = q_from_workload(w)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
                      sm_count=sm_count, ctas_per_sm=ctas_per_sm, max_splits=max_splits, margin=margin,
                      causal=w.causal, impl=impl, kv_stages=kv_stages, with_lse=True, q_mode=q_mode)
    odt = torch.bfloat16 if out_dtype is None else out_dtype
    if out_strided:  # O rows inside a wider buffer (like a fused QKV/O layout)
        big = torch.full((w.num_seqs * w.q_len, w.h_q + 8, w.d + 64), SENTINEL, dtype=odt, device="cuda")
        out = big[:, 4:4 + w.h_q, :w.d]
    else:
        out = torch.full((w.num_seqs * w.q_len, w.h_q, w.d), SENTINEL, dtype=odt, device="cuda")
    lens = w.seq_lens if plan_lens is None else plan_lens
    info = step.plan(lens, w.num_seqs)
    step.lse.fill_(SENTINEL)
    for _ in range(steps):
        step.run(q, out, kv, w.num_seqs, w.softmax_scale)
    torch.cuda.synchronize()
    status = mj_workspace_status(step.workspace)
    return {
        "out": out.float().cpu().numpy(),
        "lse": step.lse.cpu().numpy()[: w.num_seqs],
        "q_codes": step.q_codes.cpu().numpy()[: w.num_seqs],
        "q_descale": step.q_descale.cpu().numpy()[: w.num_seqs],
        "info": info,
        "status": status,
        "step": step,
    }


def run_oracle(w, units=None, q_mode="fp8"):
    codes, desc = oracle_quantize_q(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d, w.q_mul)
    qin = codes
    if q_mode == "bf16":  # the values as is, in the same packed row order
        from oracle.qquant import pack_q_rows

        qin = pack_q_rows(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d)
    out, lse = OA.decode_attention(qin, desc, w.logical("k"), w.logical("v"), w.k_scale, w.v_scale,
                                   w.block_table, w.seq_lens, num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q,
                                   h_k=w.h_k, d=w.d, page_size=w.page_size, kv_format=w.kv_format,
                                   softmax_scale=w.softmax_scale, causal=w.causal, o_mul=w.o_mul,
                                   units=units, q_values=(q_mode == "bf16"))
    return out, lse, codes, desc


def vmax_of(w, units):
    """max |dequantised V * o_mul| over the valid tokens of the given units."""
    vm = 0.0
    for b, g in units:
        L = int(w.seq_lens[b])
        if L <= 0:
            continue
        _, vc = OA.gather_unit(w.logical("k"), w.logical("v"), w.block_table, b, g, L, w.page_size,
                               w.kv_format)
        v = OA.decode_codes(vc, w.kv_format) * OA.descale_at(w.v_scale, b, g)
        if w.o_mul is not None:
            v = v[:, None, :] * w.o_mul[g * w.h_r:(g + 1) * w.h_r][None, :, :]
        vm = max(vm, float(np.abs(v).max()))
    return vm


def unit_rows(w, b, g):
    """(token rows, head slice) of unit (b, g) in the [B*q_len, h_q, d] output."""
    return slice(b * w.q_len, (b + 1) * w.q_len), slice(g * w.h_r, (g + 1) * w.h_r)


def compare(w, gpu_out, ref_out, units, label=""):
    """Element-wise comparison within the tolerance on the given units;
    padding requests must still hold the sentinel. Returns error stats."""
    vm = vmax_of(w, units)
    errs = []
    for b, g in units:
        rs, hs = unit_rows(w, b, g)
        got = gpu_out[rs, hs]
        if int(w.seq_lens[b]) <= 0:
            assert np.all(got == SENTINEL), f"{label}: padding request {b} was written"
            continue
        want = ref_out[rs, hs]
        assert np.all(np.isfinite(got)), f"{label}: non-finite output in unit {(b, g)}"
        errs.append(np.abs(got - want).reshape(-1))
    if not errs:
        return {"max": 0.0, "mean": 0.0, "vmax": vm}
    e = np.concatenate(errs)
    mx, mean = float(e.max()), float(e.mean())
    assert mx <= ATOL_MAX * vm, f"{label}: max|err| {mx:.3e} > {ATOL_MAX} * max|V| ({vm:.3e})"
    assert mean <= ATOL_MEAN * vm, f"{label}: mean|err| {mean:.3e} > {ATOL_MEAN} * max|V| ({vm:.3e})"
    return {"max": mx, "mean": mean, "vmax": vm}


def all_units(w):
    return [(b, g) for b in range(w.num_seqs) for g in range(w.h_k)]


def sample_units(w, n, seed=0):
    rng = np.random.default_rng(seed)
    units = all_units(w)
    idx = rng.choice(len(units), size=min(n, len(units)), replace=False)
    return [units[i] for i in sorted(idx)]
