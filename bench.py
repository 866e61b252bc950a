#!/usr/bin/env python3
"""Benchmark of one paged decode-attention step on GB300.

A step is the whole hot path over one batch: the split-KV plan (host) and
its upload, ``mj_quantize_q``, ``mj_decode_attention`` and ``mj_merge_lse``.
Default workload: the Qwen3-8B-shaped decode batch (B=64, q_len=1, 32/8
heads, D=128, page 16, every length 4096, per-KV-head e4m3 scales, HND,
16384 pages drawn from a 20000-page pool). Prints ONE JSON line.

* ``value``: effective KV GB/s = sum(seq_len) * h_k * 2 * row_bytes per step
  / device step time (CUDA events on the launching stream), inputs resident in
  HBM. The KV read per step (537 MB) is larger than the 129 MB L2, so no
  flush is needed between steps.
* ``e2e``: the same metric end to end through the C ABI from pinned host
  buffers: each step plans on the host, copies Q, seq_lens, the block table
  and the plan to the device, runs the three kernels and copies O back.
* ``roofline``: the decode kernel alone, algorithmic KV bytes per launch /
  its average CUDA-event duration, against the measured HBM copy bandwidth.
* ``cpu_baseline``: the CPU oracle timed on a bounded sample in a
  single-threaded subprocess.

``--impl reference`` times the CPU oracle itself, one (request, KV head)
unit per step. Under torchrun every rank runs an independent replica
(weak scaling); rank 0 prints.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn effective KV GB/s (% of HBM peak) and decode tokens/s per step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# knobs per workload: (ctas_per_sm, max_splits, kv_stages)
DEFAULT_KNOBS = {
    "qwen3_8b_decode": (2, 64, 6),
    "long_split": (2, 64, 6),
    "long_single": (2, 64, 6),
    "spec_verify": (4, 64, 4),
    "spec_verify_noncausal": (4, 64, 4),
    "fp6_decode": (2, 64, 6),
    "d256_decode": (2, 64, 2),
    "fp6_e3m2_decode": (2, 64, 6),
    "fp4_decode": (2, 64, 6),
    "tiny": (2, 16, 0),
}


# largest value of each cache format (the channel scales are amax / max)
FORMAT_MAX = {"fp8": 448.0, "e2m3": 7.5, "e3m2": 28.0, "e2m1": 6.0}


def kv_row_bytes(w) -> int:
    """Bytes of one (token, KV head) row of the workload's cache format."""
    return {"fp8": w.d, "e2m3": w.d * 3 // 4, "e3m2": w.d * 3 // 4, "e2m1": w.d // 2}[w.kv_format]


def kv_bytes_per_step(w) -> int:
    """The metric's algorithmic bytes: every valid token's K and V row of
    every KV head, read once."""
    import numpy as np

    return int(np.asarray(w.seq_lens, dtype=np.int64).sum()) * w.h_k * 2 * kv_row_bytes(w)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001 - absent on a box that had no measurement
        return FALLBACK_HBM_GBS, "fallback"


# Every source file a kernel is compiled from: a change to any of them makes
# the committed DRAM counters stale.
KERNEL_SOURCES = {
    "decode_tc.cu": ["decode_tc.cu", "decode_tc_e4m3.cu", "decode_tc_e2m3.cu", "decode_tc_e3m2.cu",
                     "decode_tc_e2m1.cu", "decode_tc_d256.cu", "decode_tc_kernel.cuh", "tc_ptx.cuh",
                     "mj_device.cuh", "mj_internal.h"],
    "decode_simt.cu": ["decode_simt.cu", "mj_device.cuh", "mj_internal.h"],
}


def _code_only(src: str) -> str:
    """C/CUDA source with comments removed and whitespace runs collapsed: a
    change to a comment does not change the compiled kernel or its counters.
    (The kernel sources hold no string literal with a comment marker.)"""
    import re

    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def _kernel_source_hash(name: str, read=None) -> str:
    """Hash of the code (not the comments) of every file the kernel is built from."""
    h = hashlib.sha256()
    for part in KERNEL_SOURCES.get(name, [name]):
        if read is None:
            with open(os.path.join(ROOT, "paged_fp8_decode_gb300", "csrc", part), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(part)
        data = _code_only(text).encode()
        h.update(part.encode() + b"\0" + len(data).to_bytes(8, "little") + data)
    return h.hexdigest()[:16]


def _traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel_file}:{workload}")
    except Exception:  # noqa: BLE001
        return None
    if not rec or rec.get("source_sha") != _kernel_source_hash(kernel_file):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:  # noqa: BLE001
            self.proc = None
        time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------
def _oracle_unit_seconds(w, units):
    """Time the oracle on the given (request, KV head) units: Q quantization
    of the whole batch + exact attention of each unit."""
    from oracle import attention as OA
    from oracle.qquant import quantize_q

    t0 = time.perf_counter()
    codes, desc = quantize_q(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d, w.q_mul)
    OA.decode_attention(codes, desc, w.logical("k"), w.logical("v"), w.k_scale, w.v_scale, w.block_table,
                        w.seq_lens, num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
                        page_size=w.page_size, kv_format=w.kv_format, softmax_scale=w.softmax_scale,
                        causal=w.causal, o_mul=w.o_mul, units=units)
    return time.perf_counter() - t0


def cpu_baseline_child(workload: str, budget_s: float, shard: str = "0/1"):
    """Run in a single-threaded subprocess: oracle KV GB/s on a time-bounded
    sample of the workload's units (shard ``i/n``: units i, i+n, ...)."""
    import synth

    w = synth.WORKLOADS[workload]()
    row = kv_row_bytes(w)
    si, sn = (int(v) for v in shard.split("/"))
    units = [(b, g) for b in range(w.num_seqs) for g in range(w.h_k) if w.seq_lens[b] > 0][si::sn]
    done, nbytes, t = 0, 0, 0.0
    while t < budget_s and done < len(units):
        batch = units[done:done + 8]
        t += _oracle_unit_seconds(w, batch)
        nbytes += sum(int(w.seq_lens[b]) for b, _ in batch) * 2 * row
        done += len(batch)
    print(json.dumps({"value": nbytes / t / 1e9 if t > 0 else 0.0, "units": done, "total_units": len(units),
                      "seconds": t,
                      "bytes": nbytes}))


# ----------------------------------------------------------------------------
# replicas (one process per GPU under torchrun; weak scaling)
# ----------------------------------------------------------------------------
def replica_workload(name: str, rank: int):
    """Rank r's batch: the Qwen3-8B decode batch is drawn with its own seed
    per rank (independent replicas); the other workloads are the same batch
    on every rank."""
    import synth

    if name == "qwen3_8b_decode":
        return synth.WORKLOADS[name](seed=1002 + 17 * rank)
    return synth.WORKLOADS[name]()


def max_over_ranks(x: float, dist, device) -> float:
    """The job's time is its slowest rank's: all-reduce MAX (a no-op alone)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(kv_bytes_per_rank: int, world: int, seconds_per_step: float) -> float:
    """Whole-job throughput: the KV bytes every rank streamed per step over the step time."""
    return kv_bytes_per_rank * world / seconds_per_step / 1e9


def measure_write_kv(w, dev, peak: float) -> dict:
    """The KV-cache write that precedes a decode step (mj_write_kv), timed on
    its own: a bulk write of every token of the workload's batch (up to
    262144), and the decode step's own write of one new token per request.
    Inputs are generated on the device (a kernel-only figure). Algorithmic
    bytes: the bf16 K and V rows read, the code rows written and the slots."""
    import ctypes

    import torch

    import paged_fp8_decode_gb300 as mj

    fmt = mj.KV_FORMATS[w.kv_format]
    row = kv_row_bytes(w)
    lib = mj.load_library()
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    out = {"format": w.kv_format}
    for label, n_tok in (("bulk", int(min(int(w.seq_lens.sum()), 262144))), ("decode_step", int(w.num_seqs))):
        pages = (n_tok + w.page_size - 1) // w.page_size + 64
        kv = torch.randn(2, n_tok, w.h_k, w.d, device=dev, generator=gen).to(torch.bfloat16)
        slots = torch.randperm(pages * w.page_size, device=dev, generator=gen)[:n_tok].to(torch.int64)
        pool = torch.empty(2, pages * w.page_size * w.h_k * row, dtype=torch.uint8, device=dev)
        amax = kv.float().abs().amax(dim=1)  # [2, h_k, d]
        if fmt == mj.MJ_KV_E4M3:
            scales = (amax.amax(dim=2) / 448.0).contiguous()  # per KV head
        else:
            scales = (amax / FORMAT_MAX[w.kv_format]).contiguous()  # per (KV head, channel)
        strides = (w.h_k * w.page_size * row, row, w.page_size * row)  # HND
        a = mj.mj_write_kv_args()
        a.num_tokens, a.h_k, a.d = n_tok, w.h_k, w.d
        a.key, a.value = kv[0].data_ptr(), kv[1].data_ptr()
        a.key_tok_stride, a.key_head_stride = kv[0].stride(0), kv[0].stride(1)
        a.value_tok_stride, a.value_head_stride = kv[1].stride(0), kv[1].stride(1)
        a.slot_mapping = slots.data_ptr()
        a.kv_format, a.page_size, a.num_pages = fmt, w.page_size, pages
        a.k_cache, a.v_cache = pool[0].data_ptr(), pool[1].data_ptr()
        a.k_stride_page, a.k_stride_token, a.k_stride_head = strides
        a.v_stride_page, a.v_stride_token, a.v_stride_head = strides
        a.k_scale, a.v_scale, a.scale_per_head = scales[0].data_ptr(), scales[1].data_ptr(), 1
        ref, st = ctypes.byref(a), stream.cuda_stream
        for _ in range(3):
            assert lib.mj_write_kv(ref, st) == 0
        reps = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            lib.mj_write_kv(ref, st)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / reps
        nbytes = 2 * n_tok * w.h_k * w.d * 2 + 2 * n_tok * w.h_k * row + n_tok * 8
        gbs = nbytes / (us * 1e-6) / 1e9
        out[label] = {"tokens": n_tok, "us": round(us, 3), "bytes": nbytes, "gbs": round(gbs, 1)}
        if label == "bulk":
            out[label]["roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                      "frac": round(gbs / peak, 4)}
        del kv, slots, pool
    return out


def _cpu_children(workload: str, budget_s: float, n: int):
    """n single-threaded oracle processes at once, on disjoint shards of the units."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", workload,
                               "--budget", str(budget_s), "--shard", f"{i}/{n}"],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
             for i in range(n)]
    res = []
    for pr in procs:
        out, err = pr.communicate(timeout=900)
        if pr.returncode != 0:
            raise RuntimeError(err[-300:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    return res


def measure_bf16_q(w, kv, dev, peak: float, cps: int, msplit: int) -> dict | None:
    """The decode step with bf16 Q as is (T5DecodeRunner's q_mode="bf16"):
    decode (+ merge) only, timed on its own. e4m3 KV only. The tensor-core
    kernel carries each Q value as two e4m3 terms."""
    if w.kv_format != "fp8":
        return None
    import numpy as np
    import torch

    from paged_fp8_decode_gb300 import DecodeStep, mj_decode_attention, mj_merge_lse
    from paged_fp8_decode_gb300.step import q_from_workload

    q = q_from_workload(w, dev)
    out = torch.empty(w.num_seqs * w.q_len, w.h_q, w.d, dtype=torch.bfloat16, device=dev)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, ctas_per_sm=cps,
                      max_splits=msplit, causal=w.causal, device=dev, q_mode="bf16")
    stream = torch.cuda.current_stream(dev)
    step.plan(w.seq_lens, w.num_seqs, stream)
    a = step.args(kv, out, w.num_seqs, w.softmax_scale, q=q)
    for _ in range(3):
        mj_decode_attention(a, stream)
        mj_merge_lse(a, stream)
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        mj_decode_attention(a, stream)
        mj_merge_lse(a, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / reps
    kv_bytes = int(w.seq_lens.astype(np.int64).sum()) * w.h_k * 2 * w.d
    gbs = kv_bytes / (us * 1e-6) / 1e9
    return {"kernel": "decode_tc (Q as two e4m3 terms)", "us": round(us, 2), "gbs": round(gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4)}}


def run_cpu_baseline(workload: str, budget_s: float = 10.0):
    """The oracle as it stands on the host cores: one single-threaded process
    per core at once (the aggregate rate), and one process alone."""
    cores = os.cpu_count() or 1
    try:
        many = _cpu_children(workload, budget_s, cores)
        one = _cpu_children(workload, budget_s, 1)[0]
    except Exception as e:  # noqa: BLE001
        return {"value": None, "unit": "GB/s", "cores": cores, "kind": "oracle", "error": str(e)}
    value = sum(j["value"] for j in many)
    units = sum(j["units"] for j in many)
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{units} of {sum(j['total_units'] for j in many)} "
                      f"(request, KV head) units of {workload}, split over {cores} single-threaded processes "
                      f"running at once ({budget_s:.0f} s of oracle time each): Q quantization of the batch + "
                      f"exact fp64 attention",
            "single_core": {"value": round(one["value"], 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{one['units']} units, {one['seconds']:.1f} s"}}


def reference_arm(args):
    """--impl reference: the CPU oracle, one (request, KV head) unit per step."""
    import synth

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]()
    row = kv_row_bytes(w)
    units = [(b, g) for b in range(w.num_seqs) for g in range(w.h_k) if w.seq_lens[b] > 0]
    for i in range(args.warmup):
        _oracle_unit_seconds(w, [units[i % len(units)]])
    t, nbytes, toks = 0.0, 0, 0
    for i in range(args.steps):
        b, g = units[(args.warmup + i) % len(units)]
        t += _oracle_unit_seconds(w, [(b, g)])
        nbytes += int(w.seq_lens[b]) * 2 * row
    value = nbytes / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "unit_per_step": "one (request, KV head)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} (request, KV head) units of {args.workload}, one per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def main_ours(args):
    import numpy as np
    import torch

    import synth
    from paged_fp8_decode_gb300 import (DecodeStep, mj_decode_attention, mj_merge_lse, mj_quantize_q,
                                        mj_workspace_status)
    from paged_fp8_decode_gb300.build import build
    from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_base = run_cpu_baseline(args.workload)

    build()
    w = replica_workload(args.workload, rank)
    cps, msplit, stages = DEFAULT_KNOBS.get(args.workload, (2, 64, 0))
    cps = args.ctas_per_sm or cps
    msplit = args.max_splits or msplit
    stages = args.kv_stages if args.kv_stages is not None else stages
    impl = {"auto": 0, "simt": 1, "tcgen05": 2}[args.variant]

    torch.cuda.set_device(dev)
    kv = paged_kv_from_workload(w, dev)
    q = q_from_workload(w, dev)
    out = torch.empty(w.num_seqs * w.q_len, w.h_q, w.d, dtype=torch.bfloat16, device=dev)
    step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, ctas_per_sm=cps,
                      max_splits=msplit, causal=w.causal, impl=impl, kv_stages=stages, device=dev,
                      q_mode=args.q_mode)
    stream = torch.cuda.current_stream(dev)
    info = step.plan(w.seq_lens, w.num_seqs, stream)
    a = step.args(kv, out, w.num_seqs, w.softmax_scale, q=q)
    kv_bytes = kv_bytes_per_step(w)
    tokens = int((w.seq_lens > 0).sum()) * w.q_len
    launches_per_step = (1 if args.q_mode == "fp8" else 0) + 1 + (1 if info["with_reduction"] else 0)

    def device_step(ev=None):
        if args.q_mode == "fp8":  # otherwise the decode kernel quantizes Q itself (or takes it as is)
            mj_quantize_q(q, w.num_seqs, w.q_len, w.h_k, step.q_codes, step.q_descale, q_mul=kv.q_mul,
                          stream=stream)
        if ev is not None:
            ev[0].record(stream)
        mj_decode_attention(a, stream)
        if ev is not None:
            ev[1].record(stream)
        mj_merge_lse(a, stream)

    for _ in range(max(3, args.warmup)):
        device_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()

    # ---- device-resident timed region: K whole steps, nothing between the
    # launches (an event between them would break the overlap of quantize and
    # decode) ------------------------------------------------------------------
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        start.record(stream)
        for i in range(args.steps):
            device_step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)

    # ---- the decode kernel alone (roofline), CUDA events around each launch
    n_dec = max(10, min(args.steps, 200))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dec)]
    for i in range(n_dec):
        device_step(evs[i])
    torch.cuda.synchronize(dev)
    decode_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    status = mj_workspace_status(step.workspace, stream)

    # ---- end to end through host buffers ----------------------------------
    q_host = q.cpu().pin_memory()
    lens_host = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).pin_memory()
    bt_host = torch.from_numpy(np.ascontiguousarray(w.block_table)).pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = (q_host.numel() * 2 + lens_host.numel() * 4 + bt_host.numel() * 4 + step.work_host.numel() * 4 +
           step.nsplit_host.numel() * 4)
    d2h = out_host.numel() * 2
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step():
        step.plan(w.seq_lens, w.num_seqs, stream)
        q.copy_(q_host, non_blocking=True)
        kv.seq_lens.copy_(lens_host, non_blocking=True)
        kv.block_table.copy_(bt_host, non_blocking=True)
        device_step()
        out_host.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)

    # the same step with the separate quantize launch, for comparison
    unfused = None
    if args.q_mode == "fp8_fused" and rank == 0:
        step_u = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
                            ctas_per_sm=cps, max_splits=msplit, causal=w.causal, impl=impl, kv_stages=stages,
                            device=dev)
        step_u.plan(w.seq_lens, w.num_seqs, stream)
        a_u = step_u.args(kv, out, w.num_seqs, w.softmax_scale)
        n_u = max(10, min(args.steps, 500))

        def step_unfused():
            mj_quantize_q(q, w.num_seqs, w.q_len, w.h_k, step_u.q_codes, step_u.q_descale, q_mul=kv.q_mul,
                          stream=stream)
            mj_decode_attention(a_u, stream)
            mj_merge_lse(a_u, stream)

        for _ in range(3):
            step_unfused()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n_u):
            step_unfused()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_u = e0.elapsed_time(e1) / n_u
        unfused = {"ms_per_step": round(ms_u, 5), "value": round(whole_job_gbs(kv_bytes, 1, ms_u * 1e-3), 2),
                   "unit": "GB/s", "steps": n_u, "note": "mj_quantize_q as its own launch before the decode"}

    # the KV-cache write before the step (its own measurement, outside the timed step)
    write_kv = measure_write_kv(w, dev, _peaks()[0]) if rank == 0 else None
    bf16_q = measure_bf16_q(w, kv, dev, _peaks()[0], cps, msplit) if rank == 0 else None

    # plan host time alone
    t0 = time.perf_counter()
    for _ in range(50):
        step.plan(w.seq_lens, w.num_seqs, stream)
    plan_us = (time.perf_counter() - t0) / 50 * 1e6
    torch.cuda.synchronize(dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(kv_bytes, world, ms_per_step * 1e-3)
    peak, peak_kind = _peaks()
    dec_avg_ms = sum(decode_ms) / len(decode_ms)
    achieved = kv_bytes / (dec_avg_ms * 1e-3) / 1e9
    kernel_file = "decode_tc.cu" if impl == 2 or (impl == 0 and os.path.exists(
        os.path.join(ROOT, "paged_fp8_decode_gb300", "csrc", "decode_tc.cu"))) else "decode_simt.cu"
    traffic = _traffic(kernel_file, args.workload)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/f32", "data": "synthetic",
        "config": {
            "workload": args.workload, "num_seqs": w.num_seqs, "q_len": w.q_len, "h_q": w.h_q, "h_k": w.h_k,
            "d": w.d, "page_size": w.page_size, "seq_len_total": int(w.seq_lens.sum()), "layout": w.layout,
            "kv_format": w.kv_format, "causal": w.causal, "parallelism": f"replicas{world}",
            "l2": f"inputs larger than L2: {kv_bytes / 1e6:.0f} MB of KV read per step vs 129 MB L2, no flush",
            "ctas_per_sm": cps, "max_splits": msplit, "kv_stages": stages, "variant": args.variant,
            "q_mode": args.q_mode,
            "with_reduction": info["with_reduction"], "chunk_tiles": info["chunk_tiles"],
            "num_work": info["num_work"],
        },
        "kv_bytes_per_step": kv_bytes,
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_hbm": round(100 * value / world / peak, 2),
        "tokens_per_s": round(tokens * world / (ms_per_step * 1e-3), 1),
        "plan_host_us": round(plan_us, 2),
        "clocks": clocks,
        "e2e": {"value": round(whole_job_gbs(kv_bytes, world, e2e_s / e2e_steps), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"of {peak_kind}", "kernel": kernel_file.replace(".cu", ""),
                     "decode_us": round(dec_avg_ms * 1e3, 3)},
        "cpu_baseline": cpu_base,
        "device_status": status,
        "write_kv": write_kv,
        "unfused_step": unfused,
        "bf16_q": bf16_q,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_decode")
    ap.add_argument("--variant", default="auto", choices=["auto", "simt", "tcgen05"])
    ap.add_argument("--q-mode", default="fp8_fused", choices=["fp8", "fp8_fused", "bf16"],
                    help="fp8: mj_quantize_q then decode; fp8_fused: the same quantization inside the "
                         "decode kernel (bit-identical output); bf16: Q as is")
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--max-splits", type=int, default=0)
    ap.add_argument("--kv-stages", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", default=None)
    ap.add_argument("--budget", type=float, default=10.0)
    ap.add_argument("--shard", default="0/1")
    args = ap.parse_args()
    if args.cpu_baseline_child:
        cpu_baseline_child(args.cpu_baseline_child, args.budget, args.shard)
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    main_ours(args)


if __name__ == "__main__":
    main()
