"""Host arithmetic of bench.py, on the CPU.

The metric's numerator is the algorithmic KV bytes of a step: every valid
token's K and V row of every KV head, read once. Pinned here against byte
counts worked out by hand for each workload, and against the oracle's own
count. Also checked: the whole-job throughput over ranks, and that a
DRAM-traffic record taken on other kernel sources is not reported.
"""

from types import SimpleNamespace

import numpy as np
import pytest

import bench
from oracle import attention as OA


def _w(lens, h_k, d, kv_format):
    return SimpleNamespace(seq_lens=np.asarray(lens, dtype=np.int32), h_k=h_k, d=d, kv_format=kv_format)


# (lengths, KV heads, head size, format, bytes worked out by hand)
CASES = {
    "tiny": ([37, 100], 2, 128, "fp8", (37 + 100) * 2 * 2 * 128),                  # 70,144
    "qwen3_8b_decode": ([4096] * 64, 8, 128, "fp8", 536_870_912),                   # 64*4096*8*256
    "long_single": ([131072], 8, 128, "fp8", 268_435_456),                          # 2^17*8*256
    "fp6_decode": ([8192] * 128, 8, 128, "e2m3", 1_610_612_736),                    # rows of 96 B
    "fp6_e3m2_decode": ([8192] * 128, 8, 128, "e3m2", 1_610_612_736),
    "fp4_decode": ([8192] * 128, 8, 128, "e2m1", 1_073_741_824),                    # rows of 64 B
    "d256_decode": ([4096] * 64, 8, 256, "fp8", 1_073_741_824),                     # rows of 256 B
    "spec_verify_padding": ([1024, 0, 16384, 0], 8, 128, "fp8", (1024 + 16384) * 8 * 256),
}


@pytest.mark.parametrize("name", list(CASES))
def test_kv_bytes_per_step(name):
    lens, h_k, d, fmt, want = CASES[name]
    w = _w(lens, h_k, d, fmt)
    assert bench.kv_bytes_per_step(w) == want
    assert OA.effective_kv_bytes(lens, h_k, d, fmt) == want


def test_row_bytes_per_format():
    assert [bench.kv_row_bytes(_w([1], 1, 128, f)) for f in ("fp8", "e2m3", "e3m2", "e2m1")] == [128, 96, 96, 64]
    assert [bench.kv_row_bytes(_w([1], 1, 256, f)) for f in ("fp8", "e2m3", "e3m2", "e2m1")] == [256, 192, 192, 128]


def test_whole_job_throughput():
    # two replicas of 536,870,912 B each in 100 us: 10,737.4 GB/s
    assert bench.whole_job_gbs(536_870_912, 2, 100e-6) == pytest.approx(10737.41824)
    assert bench.whole_job_gbs(536_870_912, 1, 85.8e-6) == pytest.approx(6257.24, rel=1e-5)


def test_traffic_record_of_other_sources_is_not_reported(monkeypatch):
    real = bench._traffic("decode_tc.cu", "qwen3_8b_decode")
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda name: "0000000000000000")
    assert bench._traffic("decode_tc.cu", "qwen3_8b_decode") is None
    assert real is None or real > 536_870_912  # DRAM bytes include the algorithmic ones


def test_source_hash_follows_code_not_comments():
    import os

    csrc = os.path.join(bench.ROOT, "paged_fp8_decode_gb300", "csrc")

    def read(part, edit=None):
        text = open(os.path.join(csrc, part), encoding="utf-8").read()
        return edit(text) if edit and part == "decode_tc_kernel.cuh" else text

    base = bench._kernel_source_hash("decode_tc.cu")
    assert bench._kernel_source_hash("decode_tc.cu", read=read) == base
    commented = lambda t: "// a new comment\n/* and a block\n   comment */\n" + t.replace("\n", "\n  ", 3)
    assert bench._kernel_source_hash("decode_tc.cu", read=lambda p: read(p, commented)) == base
    recoded = lambda t: t.replace("constexpr float kTau = 0.6f;", "constexpr float kTau = 0.5f;")
    assert "constexpr float kTau = 0.6f;" in read("decode_tc_kernel.cuh")
    assert bench._kernel_source_hash("decode_tc.cu", read=lambda p: read(p, recoded)) != base


def test_launcher_runs_n_ranks_of_this_script():
    cmd = bench.launcher_cmd(["--gpus", "4", "--steps", "10"], 4, 29512)
    i = cmd.index("torch.distributed.run")
    assert cmd[i - 1] == "-m"
    assert cmd[cmd.index("--nproc-per-node") + 1] == "4" and cmd[cmd.index("--nnodes") + 1] == "1"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1" and cmd[cmd.index("--master-port") + 1] == "29512"
    assert cmd[-4:] == [bench.__file__.replace(".pyc", ".py"), "--gpus", "4", "--steps", "10"][-4:]
    assert cmd[-5].endswith("bench.py")


def test_more_gpus_than_visible_fail_loudly(monkeypatch):
    import argparse

    import torch

    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(torch.cuda, "device_count", lambda: 1)
    args = argparse.Namespace(gpus=2)
    with pytest.raises(SystemExit) as e:
        bench.main_ours(args)
    assert "only 1 GPU" in str(e.value)


def test_world_size_must_match_gpus(monkeypatch):
    import argparse

    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as e:
        bench.main_ours(argparse.Namespace(gpus=4))
    assert "WORLD_SIZE=2" in str(e.value)
