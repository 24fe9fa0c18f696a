"""The multi-process host path of the benchmark on CPU: two gloo ranks.

The decode shards with no collective (every (sequence, KV head) is
independent), so several GPUs run independent replicas. What remains on the
host: the process-group setup from the launcher's environment, the barriers
around the timed region, the max over ranks of the measured time, the
whole-job value, and the reference arm, which runs on rank 0 only.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, port: int, q):
    # CPU ranks: with no visible GPU the bench picks gloo (two NCCL ranks
    # would need two GPUs)
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from bit_kv_cache_13_gb300 import inputs
    try:
        world, r, local = bench.dist_setup()
        bench.barrier(world)
        # rank 1 is the slower one: the job's time is its time
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        bench.barrier(world)
        spec = inputs.SPECS["qwen8b"]
        cfg = bench.config_dict(spec, None, world, l2="-")
        bytes_step = 1_000_000
        value = world * bytes_step / (slowest * 1e-3) / 1e9     # whole-job GB/s, as the bench forms it
        q.put((rank, world, r, local, dist.get_backend(), slowest, cfg["global_batch"], cfg["parallelism"], value))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, (r0, world, r, local, backend, slowest, gbatch, par, value) in enumerate(got):
        assert (r0, world, r, local, backend) == (rank, 2, rank, rank, "gloo")
        assert slowest == 15.0                      # max over ranks
        assert gbatch == 2 and par == "replicas x2"  # batch 1 per replica
        assert abs(value - 2 * 1e6 / 15e-3 / 1e9) < 1e-12


def _reference_rank(rank: int, port: int, q):
    # CPU ranks: with no visible GPU the bench picks gloo (two NCCL ranks
    # would need two GPUs)
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import argparse
    import contextlib
    import io

    import torch.distributed as dist

    import bench
    try:
        world, r, local = bench.dist_setup()
        calls = []
        bench.OracleSample = lambda *a, **k: calls.append(a) or (_ for _ in ()).throw(RuntimeError("stop"))
        args = argparse.Namespace(workload="qwen8b", warmup=0, steps=1, gpus=2)
        out = io.StringIO()
        raised = False
        with contextlib.redirect_stdout(out):
            try:
                bench.run_reference(args, world, r)
            except RuntimeError:
                raised = True
        q.put((rank, raised, len(calls), out.getvalue()))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm's work and its line belong to rank 0;
    rank 1 returns without touching the oracle (the oracle is replaced by a
    stub that stops at once, so no sample is computed)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reference_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got[0][:3] == (0, True, 1)     # rank 0 builds the oracle sample
    assert got[1] == (1, False, 0, "")    # rank 1: no oracle, no output
