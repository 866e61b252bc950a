"""The multi-process (N > 1) host path of bench.py, on CPU with gloo.

bench.py under torchrun runs one independent replica per rank (weak
scaling): rank r draws its own batch, plans it through the C ABI, times it,
and the job's time is the slowest rank's (all-reduce MAX); rank 0 reports
the whole-job throughput. Two gloo ranks run those pieces here: distinct
batches per rank, plans bit-identical to the oracle on each rank, the MAX
reduction seen identically by both ranks, and the whole-job value."""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import paged_fp8_decode_gb300 as mj
        from oracle import plan as OP

        w = bench.replica_workload("qwen3_8b_decode", rank)
        # the plan of this rank's batch through the C ABI == the oracle's plan
        got = mj.mj_plan_split_kv(w.seq_lens, w.num_seqs, w.q_len, w.h_q, w.h_k, 152, 2, 64, 0, 64)
        ref = OP.plan_split_kv(list(w.seq_lens), w.num_seqs, w.q_len, w.h_q, w.h_k, 152, 2, 64, 0, 64)
        assert np.array_equal(np.asarray(got["work"]), np.asarray(ref.work, dtype=np.int32))
        assert got["with_reduction"] == ref.with_reduction and got["chunk_tiles"] == ref.chunk_tiles
        # a per-rank "elapsed time"; the job's is the slowest rank's
        mine = 10.0 + 5.0 * rank
        slowest = bench.max_over_ranks(mine, dist, "cpu")
        kv_bytes = int(w.seq_lens.astype(np.int64).sum()) * w.h_k * 2 * w.d
        value = bench.whole_job_gbs(kv_bytes, world, slowest * 1e-3)
        # the batch differs per rank (independent replicas): compare a fingerprint
        fp = torch.tensor([float(w.block_table.reshape(-1)[:64].astype(np.int64).sum())], dtype=torch.float64)
        fps = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(fps, fp)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([slowest, value, kv_bytes] + [float(f.item()) for f in fps]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    from paged_fp8_decode_gb300.build import build

    build()
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    # both ranks see the slowest rank's time (rank 1: 15 ms)
    assert r0[0] == r1[0] == 15.0
    # whole-job value = all ranks' KV bytes over the slowest time
    assert r0[1] == pytest.approx(r0[2] * world / 15e-3 / 1e9)
    # independent replicas: rank 0 and rank 1 drew different batches
    assert r0[3] != r0[4] and np.array_equal(r0[3:], r1[3:])


def test_single_process_needs_no_collective():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbs(8_000_000_000, 1, 1.0) == 8.0
