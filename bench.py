#!/usr/bin/env python3
"""Benchmark of one paged decode-attention step on GB300.

A step is the whole hot path over one batch: the split-KV plan (host) and
its upload, Q quantization (inside the decode kernel by default, or
``mj_quantize_q`` with ``--q-mode fp8``), ``mj_decode_attention`` and
``mj_merge_lse``. Default workload: the Qwen3-8B-shaped decode batch (B=64,
q_len=1, 32/8 heads, D=128, page 16, every length 4096, per-KV-head e4m3
scales, HND, 16384 pages drawn from a 20000-page pool). Prints ONE JSON line.

* ``value``: effective KV GB/s = sum(seq_len) * h_k * 2 * row_bytes per step
  / device step time (CUDA events on the launching stream), inputs resident in
  HBM. The KV read per step (537 MB) is larger than the 129 MB L2, so no
  flush is needed between steps.
* ``configs``: the same figures for the other workloads (long-context split
  and single sequence, speculative verify causal and non-causal, packed fp6),
  each timed over a fixed number of steps of its own, with the decode kernel
  alone timed as back-to-back decode launches between two events.
* ``e2e``: the same metric end to end through the C ABI from pinned host
  buffers: every step plans on the host, uploads its inputs (Q, seq_lens,
  block table) and its plan, runs the kernels and copies O back to pinned
  host memory, where the host reads it. Two sets of buffers, each replaying
  one captured CUDA graph of that device work on its own stream, let
  consecutive steps overlap (a serving loop's pipelining).
* ``roofline``: the kernel the dispatch runs (``mj_decode_kernel``), KV
  bytes per launch / the average duration of back-to-back decode launches,
  against the measured HBM copy bandwidth.
* ``cpu_baseline``: the CPU oracle timed on a bounded sample of the units,
  one single-threaded process per host core at once (and one alone).

``--impl reference`` times the CPU oracle itself, one (request, KV head)
unit per step. ``--gpus N`` runs N independent replicas (weak scaling), one
process per GPU: under torchrun directly, else the script starts torchrun
itself; rank 0 prints.
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
    "long_split": (4, 64, 6),  # planned for four CTAs an SM, two resident: the hardware balances the second wave
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
# the workloads reported beside the headline one, and their timed steps
CONFIG_STEPS = {"long_split": 200, "long_single": 400, "spec_verify": 300, "spec_verify_noncausal": 300,
                "fp6_decode": 100}


def launcher_cmd(argv, n: int, port: int) -> list:
    """The torchrun command that runs this script as n ranks on one node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", str(n),
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def _free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _dispatch_kernel(a) -> str:
    """The decode kernel the library runs for these arguments."""
    import paged_fp8_decode_gb300 as mj

    return "decode_tc.cu" if mj.mj_decode_kernel(a) == mj.MJ_IMPL_TCGEN05 else "decode_simt.cu"


class Bench:
    """One workload resident on the device, with its step and the calls of a step."""

    def __init__(self, w, dev, knobs, q_mode: str, impl: int):
        import torch

        from paged_fp8_decode_gb300 import DecodeStep
        from paged_fp8_decode_gb300.step import paged_kv_from_workload, q_from_workload

        self.w, self.dev, self.q_mode = w, dev, q_mode
        self.cps, self.msplit, self.stages = knobs
        self.impl = impl
        self.kv = paged_kv_from_workload(w, dev)
        self.q = q_from_workload(w, dev)
        self.out = torch.empty(w.num_seqs * w.q_len, w.h_q, w.d, dtype=torch.bfloat16, device=dev)
        self.step = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
                               ctas_per_sm=self.cps, max_splits=self.msplit, causal=w.causal, impl=impl,
                               kv_stages=self.stages, device=dev, q_mode=q_mode)
        self.stream = torch.cuda.current_stream(dev)
        self.info = self.step.plan(w.seq_lens, w.num_seqs, self.stream)
        self.args = self.step.args(self.kv, self.out, w.num_seqs, w.softmax_scale, q=self.q)
        self.kv_bytes = kv_bytes_per_step(w)
        self.tokens = int((w.seq_lens > 0).sum()) * w.q_len
        self.launches = (1 if q_mode == "fp8" else 0) + 1 + (1 if self.info["with_reduction"] else 0)
        self.kernel_file = _dispatch_kernel(self.args)

    def device_step(self):
        from paged_fp8_decode_gb300 import mj_decode_attention, mj_merge_lse, mj_quantize_q

        w = self.w
        if self.q_mode == "fp8":  # otherwise the decode kernel quantizes Q itself (or takes it as is)
            mj_quantize_q(self.q, w.num_seqs, w.q_len, w.h_k, self.step.q_codes, self.step.q_descale,
                          q_mul=self.kv.q_mul, stream=self.stream)
        mj_decode_attention(self.args, self.stream)
        mj_merge_lse(self.args, self.stream)

    def time_steps(self, n: int) -> float:
        """ms per step over n back-to-back steps (CUDA events on the launching stream)."""
        import torch

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        e0.record(self.stream)
        for _ in range(n):
            self.device_step()
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / n

    def time_decode(self, n: int) -> float:
        """µs per launch of the decode kernel alone, n launches back to back
        between two events (the Q it reads was written by an earlier step)."""
        import torch

        from paged_fp8_decode_gb300 import mj_decode_attention

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        e0.record(self.stream)
        for _ in range(n):
            mj_decode_attention(self.args, self.stream)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) * 1e3 / n


def measure_config(name: str, dev, peak: float, peak_kind: str, q_mode: str, steps: int) -> dict:
    """One reported workload: step and decode-alone figures, and its DRAM traffic record."""
    import torch

    import synth
    from paged_fp8_decode_gb300 import mj_workspace_status

    w = synth.WORKLOADS[name]()
    b = Bench(w, dev, DEFAULT_KNOBS.get(name, (2, 64, 0)), q_mode, 0)
    for _ in range(5):
        b.device_step()
    ms = b.time_steps(steps)
    dec_us = b.time_decode(max(20, steps // 2))
    status = mj_workspace_status(b.step.workspace, b.stream)
    gbs = b.kv_bytes / (ms * 1e-3) / 1e9
    dec_gbs = b.kv_bytes / (dec_us * 1e-6) / 1e9
    traffic = _traffic(b.kernel_file, name)
    rec = {
        "step_us": round(ms * 1e3, 3), "kv_gbs": round(gbs, 1), "pct_of_nominal_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_hbm": round(100 * gbs / peak, 2),
        "tokens_per_s": round(b.tokens / (ms * 1e-3), 1), "decode_us": round(dec_us, 3),
        "decode_frac": round(dec_gbs / peak, 4), "kernel": b.kernel_file.replace(".cu", ""),
        "kv_bytes_per_step": b.kv_bytes, "steps": steps, "launches_per_step": b.launches,
        "knobs": {"ctas_per_sm": b.cps, "max_splits": b.msplit, "kv_stages": b.stages, "q_mode": q_mode,
                  "with_reduction": b.info["with_reduction"], "chunk_tiles": b.info["chunk_tiles"]},
        "traffic": traffic, "traffic_ratio": round(traffic / b.kv_bytes, 4) if traffic else None,
        "device_status": status,
    }
    del b, w
    torch.cuda.empty_cache()
    return rec


def e2e_pipelined(w, base, dev, knobs, q_mode: str, impl: int, n_steps: int, dist=None) -> dict:
    """The metric end to end through the C ABI from pinned host buffers.

    Every step plans on the host (mj_plan_split_kv into pinned staging),
    copies the step's inputs (bf16 Q, seq_lens, the block table: one packed
    pinned buffer, one copy) and its plan (mj_plan_upload) to the device,
    runs the kernels, copies O back to pinned host memory and reads it on the
    host. Two sets of buffers alternate, each with its own stream, and each
    set's device work (the uploads, the kernels, the download) is one CUDA
    graph captured once and replayed every step, so step n's copies and
    kernels overlap step n - 1's; the host reads step n's result two steps
    later, before it plans into that set's buffers again."""
    import numpy as np
    import torch

    from dataclasses import replace

    import paged_fp8_decode_gb300 as mj
    from paged_fp8_decode_gb300 import DecodeStep
    from paged_fp8_decode_gb300.step import q_from_workload

    q0 = q_from_workload(w, "cpu")
    cps, msplit, stages = knobs
    qb = q0.numel() * 2
    lb = w.num_seqs * 4
    bb = w.block_table.size * 4

    def al(n):
        return (n + 255) // 256 * 256

    off_l, off_b = al(qb), al(qb) + al(lb)
    nbytes = off_b + bb
    # the step's inputs, packed in one pinned host buffer (one copy per step)
    host_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    host_in[:qb].copy_(q0.view(torch.uint8).reshape(-1))
    host_in[off_l:off_l + lb].copy_(torch.from_numpy(np.ascontiguousarray(w.seq_lens)).view(torch.uint8))
    host_in[off_b:off_b + bb].copy_(torch.from_numpy(np.ascontiguousarray(w.block_table)).view(torch.uint8).reshape(-1))
    lens_np = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    slots = []
    for k in range(2):
        stream = torch.cuda.Stream(dev)
        dbuf = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        q = dbuf[:qb].view(torch.bfloat16).view(q0.shape)
        # the resident cache and scales, with this set's seq_lens and block table
        kv = replace(base, seq_lens=dbuf[off_l:off_l + lb].view(torch.int32),
                     block_table=dbuf[off_b:off_b + bb].view(torch.int32).view(w.block_table.shape))
        out = torch.empty(w.num_seqs * w.q_len, w.h_q, w.d, dtype=torch.bfloat16, device=dev)
        st = DecodeStep(max_num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d, ctas_per_sm=cps,
                        max_splits=msplit, causal=w.causal, impl=impl, kv_stages=stages, device=dev, q_mode=q_mode)
        slots.append({"stream": stream, "dbuf": dbuf, "q": q, "kv": kv, "out": out, "step": st,
                      "out_host": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                      "done": torch.cuda.Event(), "pending": False, "graph": torch.cuda.CUDAGraph()})

    def host_plan(sl):
        st = sl["step"]
        return mj.mj_plan_split_kv(lens_np, w.num_seqs, w.q_len, w.h_q, w.h_k, st.sm_count, st.ctas_per_sm,
                                   st.max_splits, st.margin, st.pad_to, work_out=st.work_host,
                                   n_splits_out=st.nsplit_host)

    def device_work(sl, info):
        st, s_ = sl["step"], sl["stream"]
        sl["dbuf"].copy_(host_in, non_blocking=True)
        mj.mj_plan_upload(st.work_host, st.nsplit_host, st.work_dev, st.nsplit_dev, st.pad_to, w.num_seqs, s_)
        st.plan_info = dict(info, num_seqs=w.num_seqs)
        a = st.args(sl["kv"], sl["out"], w.num_seqs, w.softmax_scale, q=sl["q"])
        if q_mode == "fp8":
            mj.mj_quantize_q(sl["q"], w.num_seqs, w.q_len, w.h_k, st.q_codes, st.q_descale, q_mul=sl["kv"].q_mul,
                             stream=s_)
        mj.mj_decode_attention(a, s_)
        mj.mj_merge_lse(a, s_)
        sl["out_host"].copy_(sl["out"], non_blocking=True)

    # one eager step per set (first-call set-up happens outside the graphs),
    # then the capture of each set's device work
    for sl in slots:
        info = host_plan(sl)
        with torch.cuda.stream(sl["stream"]):
            device_work(sl, info)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(sl["graph"], stream=sl["stream"]):
            device_work(sl, info)
        torch.cuda.synchronize(dev)
    reads = []

    def read(sl):
        sl["done"].synchronize()
        reads.append(float(sl["out_host"][0, 0, 0]))  # the host reads the step's result
        sl["pending"] = False

    def one(n):
        sl = slots[n & 1]
        if sl["pending"]:
            read(sl)  # step n - 2's result, before this set's buffers are reused
        host_plan(sl)
        with torch.cuda.stream(sl["stream"]):
            sl["graph"].replay()
        sl["done"].record(sl["stream"])
        sl["pending"] = True

    def drain():
        for sl in slots:
            if sl["pending"]:
                read(sl)

    for n in range(4):
        one(n)
    drain()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for n in range(n_steps):
        one(n)
    drain()
    elapsed = max_over_ranks(time.perf_counter() - t0, dist, dev)
    assert all(math.isfinite(v) for v in reads), "non-finite result read back"
    plan_h2d = slots[0]["step"].work_host.numel() * 4 + w.num_seqs * 4
    return {"seconds": elapsed, "steps": n_steps, "h2d_bytes_per_step": int(nbytes + plan_h2d),
            "d2h_bytes_per_step": int(slots[0]["out_host"].numel() * 2)}


def main_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N replicas, one process per GPU: start torchrun with this command line
        import torch

        have = torch.cuda.device_count()
        if have < args.gpus:
            raise SystemExit(f"--gpus {args.gpus}: only {have} GPU(s) visible")
        r = subprocess.run(launcher_cmd(sys.argv[1:], args.gpus, _free_port()))
        raise SystemExit(r.returncode)
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")

    import torch

    from paged_fp8_decode_gb300 import MJ_IMPL_SIMT, mj_workspace_status
    from paged_fp8_decode_gb300.build import build

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
    torch.cuda.set_device(dev)
    peak, peak_kind = _peaks()
    w = replica_workload(args.workload, rank)
    cps, msplit, stages = DEFAULT_KNOBS.get(args.workload, (2, 64, 0))
    knobs = (args.ctas_per_sm or cps, args.max_splits or msplit, args.kv_stages if args.kv_stages is not None else stages)
    impl = {"auto": 0, "simt": MJ_IMPL_SIMT, "tcgen05": 2}[args.variant]
    b = Bench(w, dev, knobs, args.q_mode, impl)

    for _ in range(max(3, args.warmup)):
        b.device_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()

    # ---- device-resident timed region: K whole steps back to back ----------
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        start.record(b.stream)
        for _ in range(args.steps):
            b.device_step()
        stop.record(b.stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)

    # ---- the decode kernel alone (roofline): back-to-back launches ---------
    dec_us = b.time_decode(max(20, min(args.steps, 400)))
    status = mj_workspace_status(b.step.workspace, b.stream)

    # ---- end to end through host buffers, pipelined ------------------------
    e2e = e2e_pipelined(w, b.kv, dev, knobs, args.q_mode, impl, max(20, min(args.steps, 400)), dist)

    # the same step with the separate quantize launch, for comparison
    unfused = None
    if args.q_mode == "fp8_fused" and rank == 0:
        bu = Bench(w, dev, knobs, "fp8", impl)
        for _ in range(3):
            bu.device_step()
        n_u = max(10, min(args.steps, 500))
        ms_u = bu.time_steps(n_u)
        unfused = {"ms_per_step": round(ms_u, 5), "value": round(whole_job_gbs(b.kv_bytes, 1, ms_u * 1e-3), 2),
                   "unit": "GB/s", "steps": n_u, "note": "mj_quantize_q as its own launch before the decode"}
        del bu

    # the KV-cache write before the step (its own measurement, outside the timed step)
    write_kv = measure_write_kv(w, dev, peak) if rank == 0 else None
    bf16_q = measure_bf16_q(w, b.kv, dev, peak, knobs[0], knobs[1]) if rank == 0 else None

    # plan host time alone
    t0 = time.perf_counter()
    for _ in range(50):
        b.step.plan(w.seq_lens, w.num_seqs, b.stream)
    plan_us = (time.perf_counter() - t0) / 50 * 1e6
    torch.cuda.synchronize(dev)

    # the other workloads (one GPU, rank 0 of a single-process run)
    configs = None
    if world == 1 and not args.no_configs:
        configs = {}
        for name, n in CONFIG_STEPS.items():
            if name != args.workload:
                configs[name] = measure_config(name, dev, peak, peak_kind, args.q_mode, n)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(b.kv_bytes, world, ms_per_step * 1e-3)
    achieved = b.kv_bytes / (dec_us * 1e-6) / 1e9
    traffic = _traffic(b.kernel_file, args.workload)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/f32", "data": "synthetic",
        "config": {
            "workload": args.workload, "num_seqs": w.num_seqs, "q_len": w.q_len, "h_q": w.h_q, "h_k": w.h_k,
            "d": w.d, "page_size": w.page_size, "seq_len_total": int(w.seq_lens.sum()), "layout": w.layout,
            "kv_format": w.kv_format, "causal": w.causal, "parallelism": f"replicas{world}",
            "l2": f"inputs larger than L2: {b.kv_bytes / 1e6:.0f} MB of KV read per step vs 129 MB L2, no flush",
            "ctas_per_sm": knobs[0], "max_splits": knobs[1], "kv_stages": knobs[2], "variant": args.variant,
            "q_mode": args.q_mode,
            "with_reduction": b.info["with_reduction"], "chunk_tiles": b.info["chunk_tiles"],
            "num_work": b.info["num_work"],
        },
        "kv_bytes_per_step": b.kv_bytes,
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_hbm": round(100 * value / world / peak, 2),
        "tokens_per_s": round(b.tokens * world / (ms_per_step * 1e-3), 1),
        "plan_host_us": round(plan_us, 2),
        "clocks": clocks,
        "e2e": {"value": round(whole_job_gbs(b.kv_bytes, world, e2e["seconds"] / e2e["steps"]), 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"], "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "steps": e2e["steps"], "ms_per_step": round(e2e["seconds"] / e2e["steps"] * 1e3, 4),
                "note": "every step plans on the host, uploads its inputs and plan, runs, downloads O and is read "
                        "on the host; two buffer sets, each replaying one captured CUDA graph of its uploads, "
                        "kernels and download on its own stream, so consecutive steps overlap"},
        "gpu_launches": b.launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"of {peak_kind}", "kernel": b.kernel_file.replace(".cu", ""),
                     "decode_us": round(dec_us, 3),
                     "timing": "back-to-back decode launches between two events"},
        "cpu_baseline": cpu_base,
        "device_status": status,
        "configs": configs,
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
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
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
