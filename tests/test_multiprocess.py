"""The N > 1 path of the benchmark on CPU: world size 2 over gloo.

The projection path does not shard (rows are independent and each GPU runs
its own replica of the block), so the only cross-rank step is the timing
reduction: every rank reports its own time, all of them take the slowest, and
the whole-job throughput counts every rank's block.  The reference arm runs
on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (ms, bench.whole_job_tflops(1e12, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo_world2():
    world = 2
    times = [3.0, 5.5]
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, times, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 5.5
    # 2 ranks x 1 TFLOP each in 5.5 ms
    assert res[0][1] == pytest.approx(2 * 1e12 / 5.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25
    assert bench.whole_job_tflops(2e12, 1, 2.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_without_work():
    a = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert bench.reference_arm(a, rank=1, world=2) == 0
