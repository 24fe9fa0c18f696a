"""The multi-process host paths on CPU: two gloo ranks.

The decode shards with no collective (every (sequence, KV head) is
independent): the benchmark runs independent replicas, and a decode can be
cut by KV head or by sequence (bit_kv_cache_13_gb300.shard).  Covered here:
the process-group setup from the launcher's environment, the barriers around
the timed region, the max over ranks of the measured time, the whole-job
value, the reference arm on rank 0 only, and two ranks that each decode one
KV-head shard (with the fp64 oracle) whose gathered outputs equal the
unsharded decode exactly.
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


# --------------------------------------------------------------- head shards

def _shard_rank(rank, world, port, q):
    """Each rank decodes its KV-head shard of one small workload with the
    fp64 oracle; the shards are gathered and rank 0 checks the concatenation
    against the unsharded oracle decode."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from bit_kv_cache_13_gb300 import inputs, shard
    from oracle import int2

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        spec = inputs.small_spec("gloo_shard", h_q=8, h_kv=4, batch=1, ctx=70)
        pos = torch.arange(spec.ctx)
        k = inputs.gen_keys(spec, 0, 0, pos).float().numpy()
        v = inputs.gen_values(spec, 0, 0, spec.ctx).float().numpy()
        mu = inputs.key_centre(torch.as_tensor(k).to(torch.bfloat16)).numpy()
        rk = np.stack([inputs.head_rotation(128, spec.name, 0, h, "Rk") for h in range(4)]).astype(np.float32)
        rv = np.stack([inputs.head_rotation(128, spec.name, 0, h, "Rv") for h in range(4)]).astype(np.float32)
        qq = inputs.gen_queries(spec, 0).double().numpy()
        bt = inputs.block_tables(spec).numpy()
        slots = np.array([bt[0, t // 16] * 16 + t % 16 for t in range(spec.ctx)])
        h0, h1 = shard.ranges(4, world)[rank]
        cache = int2.new_cache(int(bt.max()) + 1, h1 - h0)
        int2.append(cache, k[:, h0:h1], v[:, h0:h1], slots, mu[h0:h1], rk[h0:h1], rv[h0:h1])
        mine = int2.decode(qq[:, 2 * h0:2 * h1], cache, bt, [spec.ctx], mu[h0:h1], rk[h0:h1], rv[h0:h1], 0.0884, h1 - h0)
        parts = [None] * world
        dist.all_gather_object(parts, (h0, mine))
        if rank == 0:
            got = np.concatenate([p for _, p in sorted(parts, key=lambda t: t[0])], axis=1)
            full_cache = int2.new_cache(int(bt.max()) + 1, 4)
            int2.append(full_cache, k, v, slots, mu, rk, rv)
            want = int2.decode(qq, full_cache, bt, [spec.ctx], mu, rk, rv, 0.0884, 4)
            q.put(bool(np.array_equal(got, want)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_each_decode_one_head_shard():
    import multiprocessing as mp
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=10) is True


def test_shard_ranges():
    from bit_kv_cache_13_gb300 import shard
    assert shard.ranges(8, 2) == [(0, 4), (4, 8)]
    assert shard.ranges(8, 3) == [(0, 3), (3, 6), (6, 8)]
    assert shard.ranges(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    assert shard.ranges(0, 2) == [(0, 0), (0, 0)]
    for n in range(0, 20):
        for parts in range(1, 7):
            r = shard.ranges(n, parts)
            assert r[0][0] == 0 and r[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
            sizes = [b - a for a, b in r]
            assert max(sizes) - min(sizes) <= 1
