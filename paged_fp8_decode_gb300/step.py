"""One decode step through the C ABI, with the buffers a caller keeps.

:class:`DecodeStep` owns what the runner page's ``T5DecodeRunner`` keeps
between steps (``__init__``: persistent, fixed-address plan buffers, the
partial/workspace area sized by slots, the packed-Q buffer and its
descales) and issues the four calls of a step: ``plan`` (host plan plus a
pinned, asynchronous copy into the fixed device buffers, mj_plan_upload), then
``mj_quantize_q``, ``mj_decode_attention`` and ``mj_merge_lse`` on one
stream. It holds no arithmetic of its own.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (KV_FORMATS, MJ_IMPL_AUTO, mj_decode_args, mj_decode_attention, mj_merge_lse,
               mj_plan_split_kv, mj_plan_upload, mj_quantize_q, mj_slots, mj_workspace_init, mj_workspace_size)


@dataclass
class PagedKV:
    """A paged K/V cache in device memory, as the decode call sees it."""

    k_cache: torch.Tensor  # uint8 buffer
    v_cache: torch.Tensor
    k_strides: tuple  # (page, token, head) in bytes
    v_strides: tuple
    page_size: int
    num_pages: int
    kv_format: str  # "fp8" | "e2m3" | "e3m2" | "e2m1"
    k_descale: torch.Tensor  # float32
    v_descale: torch.Tensor
    descale_strides: tuple  # (seq, head) in elements
    block_table: torch.Tensor  # int32 [B, max_blocks]
    seq_lens: torch.Tensor  # int32 [B]
    q_mul: torch.Tensor | None = None  # float32 [h_q, d]
    o_mul: torch.Tensor | None = None


class DecodeStep:
    def __init__(self, *, max_num_seqs: int, q_len: int, h_q: int, h_k: int, d: int = 128,
                 sm_count: int | None = None, ctas_per_sm: int = 2, max_splits: int = 16,
                 margin: int = 0, causal: bool = True, impl: int = MJ_IMPL_AUTO, kv_stages: int = 0,
                 evict_first: bool = True, device="cuda", with_lse: bool = False, q_mode: str = "fp8"):
        """``q_mode``: "fp8" (dynamic e4m3 Q, mj_quantize_q in the step),
        "fp8_fused" (the same quantization done by the decode kernel; the
        step is decode + merge) or "bf16" (Q as is; decode + merge)."""
        assert q_mode in ("fp8", "fp8_fused", "bf16")
        self.q_mode = q_mode
        self.device = torch.device(device)
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.max_num_seqs, self.q_len, self.h_q, self.h_k, self.d = max_num_seqs, q_len, h_q, h_k, d
        self.h_r = h_q // h_k
        self.n_q = q_len * self.h_r
        self.sm_count, self.ctas_per_sm, self.max_splits = sm_count, ctas_per_sm, max_splits
        self.margin, self.causal = margin, causal
        self.impl, self.kv_stages, self.evict_first = impl, kv_stages, evict_first
        self.slots = mj_slots(sm_count, ctas_per_sm, h_k, q_len, h_q)
        self.pad_to = max(self.slots, max_num_seqs)
        dev = self.device
        # fixed-address device plan buffers + pinned host staging
        self.work_dev = torch.zeros(self.pad_to, 4, dtype=torch.int32, device=dev)
        self.nsplit_dev = torch.ones(max(1, max_num_seqs), dtype=torch.int32, device=dev)
        self.work_host = torch.zeros(self.pad_to, 4, dtype=torch.int32).pin_memory()
        self.nsplit_host = torch.ones(max(1, max_num_seqs), dtype=torch.int32).pin_memory()
        self._staged = None  # event after the last H2D copy of the staging buffers
        # packed Q and its descales
        self.q_codes = torch.empty(max(1, max_num_seqs), h_k, self.n_q, d, dtype=torch.uint8, device=dev)
        self.q_descale = torch.ones(max(1, max_num_seqs), h_k, dtype=torch.float32, device=dev)
        # workspace: status word + partials sized by slots
        self.ws_bytes = mj_workspace_size(self.slots, max_splits, q_len, h_q, h_k, d)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        mj_workspace_init(self.workspace)
        self.lse = (torch.empty(max(1, max_num_seqs), h_k, self.n_q, dtype=torch.float32, device=dev)
                    if with_lse else None)
        self.plan_info = None

    # ------------------------------------------------------------------ plan
    def plan(self, seq_lens_host, num_seqs: int, stream=None) -> dict:
        """Host plan into the pinned staging buffers, then an asynchronous
        copy into the fixed device buffers on ``stream``."""
        if self._staged is not None:
            self._staged.synchronize()  # the previous copy has read the staging buffers
        info = mj_plan_split_kv(np.asarray(seq_lens_host, dtype=np.int32), num_seqs, self.q_len, self.h_q,
                                self.h_k, self.sm_count, self.ctas_per_sm, self.max_splits, self.margin,
                                self.pad_to, work_out=self.work_host, n_splits_out=self.nsplit_host)
        s = stream or torch.cuda.current_stream(self.device)
        mj_plan_upload(self.work_host, self.nsplit_host, self.work_dev, self.nsplit_dev, self.pad_to, num_seqs, s)
        if self._staged is None:
            self._staged = torch.cuda.Event()
        self._staged.record(s)
        info["num_seqs"] = num_seqs
        self.plan_info = info
        return info

    # ------------------------------------------------------------- the calls
    def args(self, kv: PagedKV, out: torch.Tensor, num_seqs: int, softmax_scale: float,
             q: torch.Tensor | None = None) -> mj_decode_args:
        """The decode call's arguments; ``q`` (bf16 mode): the bf16 Q it reads."""
        for name, t in (("out", out), ("q", q), ("k_cache", kv.k_cache), ("v_cache", kv.v_cache),
                        ("k_descale", kv.k_descale), ("v_descale", kv.v_descale), ("block_table", kv.block_table),
                        ("seq_lens", kv.seq_lens), ("q_mul", kv.q_mul), ("o_mul", kv.o_mul)):
            if t is not None and not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor: the kernels read it through a device pointer")
        info = self.plan_info
        a = mj_decode_args()
        if self.q_mode in ("bf16", "fp8_fused"):
            assert q is not None and q.dtype == torch.bfloat16 and q.stride(2) == 1
            a.q_mode, a.q_bf16 = (1 if self.q_mode == "bf16" else 2), q.data_ptr()
            a.q_tok_stride, a.q_head_stride = q.stride(0), q.stride(1)
            if self.q_mode == "fp8_fused" and kv.q_mul is not None:
                a.q_mul = kv.q_mul.data_ptr()
        a.num_seqs, a.q_len, a.h_q, a.h_k, a.d = num_seqs, self.q_len, self.h_q, self.h_k, self.d
        a.causal = 1 if self.causal else 0
        a.softmax_scale = softmax_scale
        a.q_codes, a.q_descale = self.q_codes.data_ptr(), self.q_descale.data_ptr()
        a.kv_format, a.page_size, a.num_pages = KV_FORMATS[kv.kv_format], kv.page_size, kv.num_pages
        a.k_cache, a.v_cache = kv.k_cache.data_ptr(), kv.v_cache.data_ptr()
        a.k_stride_page, a.k_stride_token, a.k_stride_head = kv.k_strides
        a.v_stride_page, a.v_stride_token, a.v_stride_head = kv.v_strides
        a.k_descale, a.v_descale = kv.k_descale.data_ptr(), kv.v_descale.data_ptr()
        a.descale_seq_stride, a.descale_head_stride = kv.descale_strides
        a.block_table, a.block_table_stride = kv.block_table.data_ptr(), kv.block_table.stride(0)
        a.seq_lens = kv.seq_lens.data_ptr()
        a.work, a.n_splits = self.work_dev.data_ptr(), self.nsplit_dev.data_ptr()
        a.num_work = self.pad_to
        a.with_reduction = 1 if info["with_reduction"] else 0
        a.chunk_tiles, a.max_splits, a.part_seqs = info["chunk_tiles"], self.max_splits, self.slots
        a.o_mul = kv.o_mul.data_ptr() if kv.o_mul is not None else None
        assert out.dtype in (torch.bfloat16, torch.float16), "the decode output is bf16 or fp16"
        a.out = out.data_ptr()
        a.out_dtype = 1 if out.dtype == torch.float16 else 0
        a.out_tok_stride, a.out_head_stride = out.stride(0), out.stride(1)
        a.lse = self.lse.data_ptr() if self.lse is not None else None
        a.workspace, a.workspace_bytes = self.workspace.data_ptr(), self.ws_bytes
        a.impl, a.kv_stages, a.evict_first = self.impl, self.kv_stages, 1 if self.evict_first else 0
        return a

    def run(self, q: torch.Tensor, out: torch.Tensor, kv: PagedKV, num_seqs: int, softmax_scale: float,
            stream=None, args: mj_decode_args | None = None):
        """Quantize Q (fp8 mode), decode, merge: the device part of one step."""
        if self.q_mode == "fp8":
            mj_quantize_q(q, num_seqs, self.q_len, self.h_k, self.q_codes, self.q_descale, q_mul=kv.q_mul,
                          stream=stream)
        a = args if args is not None else self.args(kv, out, num_seqs, softmax_scale, q=q)
        mj_decode_attention(a, stream)
        mj_merge_lse(a, stream)
        return out


def paged_kv_from_workload(w, device="cuda") -> PagedKV:
    """Move a synthetic workload's cache, tables and scales to the device."""
    dev = torch.device(device)
    k = torch.from_numpy(np.ascontiguousarray(w.k_cache)).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(w.v_cache)).to(dev)
    ks = torch.from_numpy(np.ascontiguousarray(w.k_scale, dtype=np.float32)).to(dev)
    vs = torch.from_numpy(np.ascontiguousarray(w.v_scale, dtype=np.float32)).to(dev)
    ds = (0, 0) if w.k_scale.size == 1 else (0, 1)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(dev)
    sl = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(dev)
    qm = torch.from_numpy(w.q_mul).to(dev) if w.q_mul is not None else None
    om = torch.from_numpy(w.o_mul).to(dev) if w.o_mul is not None else None
    return PagedKV(k_cache=k, v_cache=v, k_strides=tuple(w.kv_strides), v_strides=tuple(w.kv_strides),
                   page_size=w.page_size, num_pages=w.num_pages, kv_format=w.kv_format, k_descale=ks,
                   v_descale=vs, descale_strides=ds, block_table=bt, seq_lens=sl, q_mul=qm, o_mul=om)


def q_from_workload(w, device="cuda") -> torch.Tensor:
    return torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).to(device)
