#!/usr/bin/env python
"""Benchmark: packed-KV decode attention over the rotated INT2 cache.

Workload (default): Qwen3-8B-shaped decode step, 36 layers x (32 q / 8 KV
heads, d = 128), batch 1, 128K context.  One step = for every layer, one
launch of kvq_decode_step_int2: the quantise-on-append of the new token and
the fused packed-cache decode attention over the 128K tokens; the 36
launches are replayed as one CUDA graph.  Inputs are synthetic and seeded;
every cache is prefilled through the library's own append call before
timing.

Prints one JSON line.  `value` is achieved algorithmic bandwidth (packed
cache bytes + q/out + new-token traffic per step / device time per step,
summed over ranks); `e2e` is the same metric through the C ABI with the
step's inputs copied from pinned host memory and its outputs copied back
inside the timed region; `roofline` is the step kernel alone (36 launches
between one pair of CUDA events); `bgtq` is the Block-GTQ K3V3 decode at
128K; `sweep70b`, `llama8b` and `tiny` are single decode launches of the
other workloads with an L2 flush before each; `cpu_baseline` is the fp64
oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import os
import argparse
import hashlib
import json
import math
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_13_gb300 import _lib, inputs  # noqa: E402
from bit_kv_cache_13_gb300.workload import BgtqLayer, Int2Layer, history_positions  # noqa: E402

METRIC = "packed-KV decode attention HBM GB/s (% of 8 TB/s) and ms/step at 128K ctx"
NOMINAL_HBM_GBS = 8000.0
TOKEN_HEAD_BYTES = 96  # K codes 32 + K scale/min 16 + V codes 32 + V scale/min 16


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash(names) -> str:
    """Hash of the kernel's code: line comments and blank lines are left out,
    so a comment edit does not retire the counters taken on that code."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "bit_kv_cache_13_gb300", "csrc", name), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, sources, per_launch_units: int):
    """dram bytes per launch from the committed ncu summary, scaled to this
    launch's token-heads; None if absent or taken on other kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_hash") != kernel_source_hash(sources):
        return None
    return int(rec["dram_bytes_per_token_head"] * per_launch_units)


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        pw = [float(r[3]) for r in rows if r[3] not in ("", "[N/A]")]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ workload

def arena(tensors, device):
    """One contiguous byte buffer holding copies of `tensors`, each 256-byte
    aligned, and views of it shaped like them: a step's host I/O is then one
    copy each way."""
    offs, n = [], 0
    for t in tensors:
        n = (n + 255) // 256 * 256
        offs.append(n)
        n += t.numel() * t.element_size()
    buf = torch.zeros(n, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class Int2Step:
    """All layers of one decode step, resident on the device; the per-step
    inputs (q, new k / v) and outputs live in one arena each.  A layer's step
    is one launch of kvq_decode_step_int2: the new token is appended at
    position ctx - 1 and the ctx tokens are attended."""

    def __init__(self, spec, device):
        self.spec = spec
        self.layers = []
        self.q, self.k_new, self.v_new, self.out, self.ws = [], [], [], [], []
        for l in range(spec.n_layers):
            layer = Int2Layer(spec, l, device=device)
            layer.prefill()
            k, v = layer.new_kv()
            self.layers.append(layer)
            self.q.append(layer.queries())
            self.k_new.append(k)
            self.v_new.append(v)
            self.out.append(torch.zeros((spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=device))
            self.ws.append(layer.workspace())
        L = spec.n_layers
        self.in_arena, views = arena(self.q + self.k_new + self.v_new, device)
        self.q, self.k_new, self.v_new = views[:L], views[L:2 * L], views[2 * L:]
        self.out_arena, self.out = arena(self.out, device)
        torch.cuda.synchronize()

    def step(self, l):
        L = self.layers[l]
        # each layer's rotations, block table and cache are written only by
        # its own step, never by the launch just before (another layer's)
        _lib.kvq_decode_step_int2(self.q[l], self.k_new[l], self.v_new[l], L.cache, L.num_pages, L.block_table,
                                  L.context_lens, L.mu, L.R_k, L.R_v, L.scale, self.out[l], self.ws[l],
                                  flags=_lib.KVQ_STEP_INPUTS_READY)

    def decode(self, l):
        L = self.layers[l]
        _lib.kvq_decode_attn_int2(self.q[l], L.cache, L.num_pages, L.block_table, L.context_lens, L.R_k, L.R_v,
                                  L.scale, self.out[l], self.ws[l])

    def run(self):
        for l in range(len(self.layers)):
            self.step(l)

    # byte accounting (algorithmic)
    def units_per_decode(self) -> int:
        return self.spec.batch * self.spec.ctx * self.spec.h_kv

    def bytes_per_decode(self) -> int:
        s = self.spec
        return self.units_per_decode() * TOKEN_HEAD_BYTES + s.batch * s.h_q * s.d * (2 + 4)

    def bytes_per_append(self) -> int:
        s = self.spec
        return s.batch * s.h_kv * (2 * s.d * 2 + TOKEN_HEAD_BYTES)

    def bytes_per_step(self) -> int:
        return self.spec.n_layers * (self.bytes_per_decode() + self.bytes_per_append())

    def host_io(self):
        """Bytes copied per step: the input and output arenas."""
        return self.in_arena.numel(), self.out_arena.numel()


def time_launches(stream, fn, n):
    """Mean duration (ms) of fn() over n launches, CUDA events around each."""
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
    stream.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def measure_int2_decode(spec, device, stream, reps, step=False):
    """One INT2 layer of `spec` decoded (kvq_decode_attn_int2, automatic split)
    or, with step=True, one fused decode step (kvq_decode_step_int2): a 256
    MB L2 flush before each timed launch, so the cache streams from HBM even
    when it would fit L2.  Returns ms per launch, GB/s of the packed cache +
    q/out and the fraction of the measured HBM bandwidth."""
    layer = Int2Layer(spec, 0, device=device)
    layer.prefill()
    q = layer.queries()
    out = torch.zeros((spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=device)
    ws = layer.workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    if step:
        k_new, v_new = layer.new_kv()
        call = lambda: _lib.kvq_decode_step_int2(q, k_new, v_new, layer.cache, layer.num_pages, layer.block_table,
                                                 layer.context_lens, layer.mu, layer.R_k, layer.R_v, layer.scale,
                                                 out, ws)
    else:
        call = lambda: _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table,
                                                 layer.context_lens, layer.R_k, layer.R_v, layer.scale, out, ws)
    for _ in range(3):
        call()
    durs = []
    for _ in range(reps):
        flush.zero_()
        durs.append(time_launches(stream, call, 1))
    ms = statistics.median(durs)
    nbytes = layer.packed_bytes_per_decode() + spec.batch * spec.h_q * spec.d * 6
    peak, _ = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    del layer
    torch.cuda.empty_cache()
    return {"batch": spec.batch, "ctx": spec.ctx, "us_per_launch": round(ms * 1e3, 2), "value": round(gbs, 2),
            "frac": round(gbs / peak, 4), "bytes": nbytes}


SWEEP70B = [(B, T) for B in (1, 8, 32, 64) for T in (4096, 32768, 131072)] + [(1, 262144), (1, 524288)]


def measure_int2_sweep70b(device, stream, reps):
    """The 70B-class GQA-8 grid (64 q / 8 KV heads, INT2 K/V): batch {1, 8,
    32, 64} x context {4K, 32K, 128K}, plus batch 1 at 256K and 512K; one
    decode launch per point, L2 flushed before each.  Points whose cache
    fits L2 many times over (batch 1 at 4K, ~3 MB) are latency-bound and
    reported, not held to the HBM roofline."""
    peak, kind = peaks()
    pts = [measure_int2_decode(inputs.sweep70b_spec(B, T), device, stream, reps) for B, T in SWEEP70B]
    return {"workload": "sweep70b: 64 q / 8 KV heads, d=128, INT2 K/V groups of 32 + fp16 scale/min, "
                        "batch x context grid", "kernel": "decode_int2_kernel<2>", "unit": "GB/s",
            "peak": peak, "peak_kind": kind, "points": pts,
            "l2": "256 MB buffer written before every timed launch"}


def measure_bgtq(device, stream, reps):
    """Block-GTQ K3V3 decode at 128K (32 q / 8 KV heads, B = 1): kernel-alone
    bandwidth of the packed stream (KB + 16 + VB + 2 bytes per token-head)."""
    spec = inputs.SPECS["bgtq"]
    layer = BgtqLayer(spec, 0, device=device)
    layer.prefill()
    k, v = layer.new_kv()
    layer.append(k, v, layer.new_slots())
    q = layer.queries()
    out = torch.zeros((spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=device)
    ws = layer.workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)   # evict the 120 MB cache from L2
    for _ in range(3):
        layer.decode(q, out, ws)
    durs = []
    for _ in range(reps):
        flush.zero_()
        durs.append(time_launches(stream, lambda: layer.decode(q, out, ws), 1))
    ms = statistics.median(durs)
    units = spec.batch * spec.ctx * spec.h_kv
    nbytes = units * layer.bytes_per_token_head() + spec.batch * spec.h_q * spec.d * 6
    peak, kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "bgtq K3V3: 32 q / 8 KV heads, batch 1, 131072 ctx, widths greedy in [1,8], sum 192",
            "kernel": "bgtq_decode_kernel", "bytes_per_token_head": layer.bytes_per_token_head(),
            "ms_per_decode": round(ms, 4), "value": round(gbs, 2), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind,
                         "traffic": profiled_traffic("bgtq_decode", ("bgtq_decode.cu", "bgtq_common.cuh", "merge.cuh", "kvq_common.cuh"),
                                                     units)},
            "l2": "256 MB buffer written before every timed launch"}


def measure_int2_window(spec, device, stream, reps):
    """INT2 decode of one 128K layer with a BF16 window of 4 sink + 128
    recent tokens per sequence (kvq_decode_attn_int2_window), against the
    plain decode of the same layer; a 256 MB L2 flush before each launch."""
    layer = Int2Layer(spec, 0, device=device)
    layer.prefill()
    q = layer.queries()
    g = torch.Generator(device=device)
    g.manual_seed(13)
    w = inputs.WINDOW_SINK + inputs.WINDOW_RECENT
    win_k = torch.randn((spec.batch, w, spec.h_kv, spec.d), generator=g, device=device).to(torch.bfloat16)
    win_v = torch.randn((spec.batch, w, spec.h_kv, spec.d), generator=g, device=device).to(torch.bfloat16)
    win_lens = torch.full((spec.batch,), w, dtype=torch.int32, device=device)
    out = torch.zeros((spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=device)
    ws = layer.workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    plain = lambda: _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                              layer.R_k, layer.R_v, layer.scale, out, ws)
    window = lambda: _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table,
                                                      layer.context_lens, layer.R_k, layer.R_v, layer.mu, win_k,
                                                      win_v, win_lens, layer.scale, out, ws)
    res = {}
    for name, fn in (("plain", plain), ("window", window)):
        for _ in range(3):
            fn()
        durs = []
        for _ in range(reps):
            flush.zero_()
            durs.append(time_launches(stream, fn, 1))
        res[name] = statistics.median(durs)
    # the packed cache, the BF16 window (keys and values), q in and out
    nbytes = (layer.packed_bytes_per_decode() + spec.batch * w * spec.h_kv * spec.d * 2 * 2
              + spec.batch * spec.h_q * spec.d * 6)
    peak, kind = peaks()
    gbs = nbytes / (res["window"] * 1e-3) / 1e9
    out_line = {"workload": f"{spec.name}: one layer, batch {spec.batch}, {spec.ctx} cached tokens + a BF16 window of "
                            f"{w} tokens (4 sink + 128 recent) per sequence",
                "kernel": "decode_int2_kernel<1, true>", "ms_per_decode": round(res["window"], 4),
                "ms_plain_decode": round(res["plain"], 4), "value": round(gbs, 2), "unit": "GB/s",
                "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                             "frac": round(gbs / peak, 4), "peak_kind": kind},
                "l2": "256 MB buffer written before every timed launch"}
    del layer
    torch.cuda.empty_cache()
    return out_line


def fp32_peak_tflops():
    """Derived fp32 fma peak of the device: 128 fp32 lanes per SM x SMs x 2
    flop per fma at the maximum SM clock (MEASURED_PEAKS.json, else 2070 MHz)."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sms} SMs x 128 fp32 lanes x 2 flop x {mhz / 1e3:.2f} GHz"


def measure_append_prefill(spec, device, stream, reps):
    """Batched prefill append: one layer's whole 128K-token history through
    kvq_append_int2 in one call (8 KV heads).  The rotation is a fixed-order
    fp32 fma chain of 128 steps per coordinate (16K fma per token-head and
    side), so the bound is fp32 fma issue, not HBM."""
    layer = Int2Layer(spec, 0, device=device)
    k, v = layer.history_kv(0)
    layer.mu = inputs.key_centre(k).to(device).contiguous()
    sl = layer.slots(0, history_positions(spec)).contiguous()
    k, v = k.contiguous(), v.contiguous()
    call = lambda: _lib.kvq_append_int2(k, v, sl, layer.mu, layer.R_k, layer.R_v, layer.cache, layer.num_pages)
    call()
    ms = statistics.median(time_launches(stream, call, 1) for _ in range(reps))
    th = k.shape[0] * spec.h_kv
    tflops = th * 2 * 2 * spec.d * spec.d / (ms * 1e-3) / 1e12
    peak_tf, peak_kind = fp32_peak_tflops()
    out = {"workload": f"{spec.name}: one layer, {k.shape[0]} tokens x {spec.h_kv} KV heads appended in one call",
           "kernel": "append_int2_prefill_kernel", "ms_per_layer": round(ms, 4),
           "value": round(th / (ms * 1e-3) / 1e6, 2), "unit": "M token-heads/s",
           "roofline": {"bound": "alu", "achieved": round(tflops, 3), "peak": round(peak_tf, 1),
                        "unit": "TFLOP/s", "frac": round(tflops / peak_tf, 4), "peak_kind": peak_kind},
           "bytes_per_token_head": {"read": 2 * 2 * spec.d, "written": 96}}
    del layer, k, v
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle

def host_cpu():
    """Host cores this process may use and the CPU model (as far as the OS says)."""
    try:
        cores = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        cores = os.cpu_count() or 1
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                break
    except OSError:
        pass
    return cores, f"{platform.machine()} {model}".strip()


class OracleSample:
    """The fp64 oracle on one (layer, KV head) of the same workload, set up
    from the seeded input generators alone (no GPU, no library).  The head's
    cache is built untimed; a step is the oracle's new-token append plus the
    decode of that head's query group over the full context."""

    def __init__(self, spec, layer_idx, h):
        from oracle import int2
        self.int2, self.spec, self.h = int2, spec, h
        d, g, T = spec.d, spec.g, spec.ctx
        pos = history_positions(spec)
        k = inputs.gen_keys(spec, layer_idx, 0, pos)
        v = inputs.gen_values(spec, layer_idx, 0, pos.numel())
        self.mu = inputs.key_centre(k).numpy()[h:h + 1]
        self.k_new = inputs.gen_keys(spec, layer_idx, 0, torch.tensor([T - 1]), tag="new")[:, h:h + 1].float().numpy()
        self.v_new = inputs.gen_values(spec, layer_idx, 0, 1, tag="new")[:, h:h + 1].float().numpy()
        self.q = inputs.gen_queries(spec, layer_idx).double().numpy()[0:1, h * g:(h + 1) * g]
        bt = inputs.block_tables(spec).numpy()
        self.bt = bt[0:1]
        self.slots = np.array([self.bt[0, t // 16] * 16 + t % 16 for t in range(T)])
        self.rk = inputs.head_rotation(d, spec.name, layer_idx, h, "Rk").astype(np.float32)[None]
        self.rv = inputs.head_rotation(d, spec.name, layer_idx, h, "Rv").astype(np.float32)[None]
        self.cache = int2.new_cache(int(bt.max()) + 1, 1)
        int2.append(self.cache, k[:, h:h + 1].float().numpy(), v[:, h:h + 1].float().numpy(), self.slots[:-1],
                    self.mu, self.rk, self.rv, exact_chain=False)
        self.label = f"layer {layer_idx} kv-head {h}"
        self.nbytes = T * TOKEN_HEAD_BYTES + g * d * 6 + (2 * d * 2 + TOKEN_HEAD_BYTES)

    def step(self) -> float:
        t0 = time.perf_counter()
        self.int2.append(self.cache, self.k_new, self.v_new, self.slots[-1:], self.mu, self.rk, self.rv)
        self.int2.decode(self.q, self.cache, self.bt, [self.spec.ctx], self.mu, self.rk, self.rv,
                         1 / math.sqrt(self.spec.d), 1)
        return time.perf_counter() - t0


def oracle_baseline(spec, seconds_target=15.0):
    """GB/s of the oracle over (layer, head) samples, ~seconds_target of work."""
    pairs = [(0, 0), (spec.n_layers - 1, spec.h_kv - 1), (spec.n_layers // 2, 3)]
    elapsed, nbytes, labels = 0.0, 0, []
    for l, h in pairs:
        smp = OracleSample(spec, l, h)
        n = 0
        while elapsed < seconds_target * (len(labels) + 1) / len(pairs) or n == 0:
            elapsed += smp.step()
            nbytes += smp.nbytes
            n += 1
        labels.append(f"{smp.label} x{n}")
    return nbytes / elapsed / 1e9, elapsed, "; ".join(labels)


# ------------------------------------------------------------------ arms

def config_dict(spec, args, world, l2):
    return {"workload": f"{spec.name}: {spec.n_layers} layers x ({spec.h_q} q / {spec.h_kv} KV heads, d={spec.d}), "
                        f"batch {spec.batch}, {spec.ctx} ctx, INT2 K/V groups of 32 + fp16 scale/min, page 16",
            "layers": spec.n_layers, "global_batch": spec.batch * world, "seq_len": spec.ctx,
            "parallelism": f"replicas x{world}", "l2": l2}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload run by the fp64 CPU oracle."""
    if rank != 0:
        return
    spec = inputs.SPECS[args.workload]
    smp = OracleSample(spec, 0, 0)
    times = []
    for i in range(args.warmup + args.steps):
        el = smp.step()
        if i >= args.warmup:
            times.append(el)
    vals = [smp.nbytes / t / 1e9 for t in times]
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.median(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(spec, args, 1, l2="oracle on host cores"),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": host_cpu()[0], "cpu": host_cpu()[1],
                         "kind": "oracle",
                         "sample": f"per step: new-token append + decode of one (layer, KV head) at {spec.ctx} "
                                   f"tokens ({smp.label}); bytes = that head's packed cache + q/out"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_extras(line, spec, device, stream):
    """The sub-measurements beside the headline step: the batched prefill
    append, the 70B-class grid (and its batch-8 128K point as `gqa8`), the
    Llama-8B-shaped decode, the tiny fused step and the BF16-window decode."""
    line["append_prefill"] = measure_append_prefill(spec, device, stream, reps=3)
    sweep = measure_int2_sweep70b(device, stream, reps=3)
    line["sweep70b"] = sweep
    g8 = next(p for p in sweep["points"] if p["batch"] == 8 and p["ctx"] == 131072)
    line["gqa8"] = {"workload": "sweep70b: 64 q / 8 KV heads, batch 8, 131072 ctx, INT2 cache",
                    "kernel": "decode_int2_kernel<2>", "ms_per_decode": round(g8["us_per_launch"] / 1e3, 4),
                    "value": g8["value"], "unit": "GB/s",
                    "roofline": {"bound": "hbm", "achieved": g8["value"], "peak": sweep["peak"], "unit": "GB/s",
                                 "frac": g8["frac"], "peak_kind": sweep["peak_kind"],
                                 "traffic": profiled_traffic("decode_int2_gqa8", ("decode_int2.cu", "int2_quant.cuh",
                                                                                   "merge.cuh", "kvq_common.cuh"),
                                                             8 * 131072 * 8)}}
    ll = measure_int2_decode(inputs.SPECS["llama8b"], device, stream, reps=5)
    line["llama8b"] = {"workload": "llama8b: 32 q / 8 KV heads, batch 8, 32768 ctx (post-RoPE keys, theta 5e5), "
                                   "INT2 cache", "kernel": "decode_int2_kernel<1>", **ll, "unit": "GB/s",
                       "l2": "256 MB buffer written before every timed launch"}
    ti = measure_int2_decode(inputs.SPECS["tiny"], device, stream, reps=10, step=True)
    line["tiny"] = {"workload": "tiny: 1 KV head, 4 q heads, batch 1, 256 cached tokens + 1 decode token, one "
                                "fused decode step", "kernel": "decode_int2_kernel<1> (step)", **ti,
                    "unit": "GB/s", "bound": "latency (24 KB of cache)",
                    "l2": "256 MB buffer written before every timed launch"}
    line["window"] = measure_int2_window(spec, device, stream, reps=5)


def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    _lib.load()
    spec = inputs.SPECS[args.workload]
    st = Int2Step(spec, device)
    stream = torch.cuda.Stream(device=device)

    # warm-up + graph capture of the whole step
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            st.run()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            st.run()
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    # ---- timed region (device time, graph replays)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("step_timed")   # lets a profiler pick out the timed launches
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(args.steps):
                graph.replay()
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    barrier(world)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world)
    ms_per_step = total_ms / args.steps
    bytes_step = st.bytes_per_step()
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9
    clocks = clk.summary()

    # ---- the step kernel alone: the 36 layers' launches back to back between
    # one pair of CUDA events (launches are enqueued faster than they run, so
    # no host gap is timed); each layer's cache is cold in L2.  The same for
    # the decode-only entry point, for comparison.
    dec_ms, only_ms = [], []
    for _ in range(max(2, min(args.steps, 5))):
        dec_ms.append(time_launches(stream, lambda: [st.step(l) for l in range(spec.n_layers)], 1) / spec.n_layers)
        only_ms.append(time_launches(stream, lambda: [st.decode(l) for l in range(spec.n_layers)], 1)
                       / spec.n_layers)
    dec_avg_ms = statistics.median(dec_ms)
    peak, peak_kind = peaks()
    achieved = (st.bytes_per_decode() + st.bytes_per_append()) / (dec_avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic("step_int2", ("decode_int2.cu", "int2_quant.cuh", "merge.cuh", "kvq_common.cuh"),
                               st.units_per_decode())

    # ---- end to end through the C ABI with host buffers
    h2d, d2h = st.host_io()
    host_in = st.in_arena.cpu().pin_memory()
    host_out = torch.empty(st.out_arena.shape, dtype=torch.uint8).pin_memory()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            st.in_arena.copy_(host_in, non_blocking=True)     # the step's q and new k / v
            graph.replay()
            host_out.copy_(st.out_arena, non_blocking=True)   # the step's outputs
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    e2e_value = world * bytes_step / (e2e_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8 codes, fp16 scale/min, fp32 softmax/accumulate", "data": "synthetic",
        "config": config_dict(spec, args, world, l2=f"inputs larger than L2: {bytes_step / 1e9:.2f} GB read per step"),
        "pct_of_8TBs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100.0 * value / world / peak, 2),
        "step_ms_median": round(statistics.median(step_ms), 4),
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "decode_int2_kernel (step: new-token append + decode)",
                     "avg_launch_us": round(dec_avg_ms * 1e3, 3),
                     "timing": "36 layer steps back to back, one event pair, median of 5",
                     "bytes_per_launch": st.bytes_per_decode() + st.bytes_per_append(),
                     "decode_only_us": round(statistics.median(only_ms) * 1e3, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": spec.n_layers * args.steps,
        "clocks": clocks,
    }
    del graph, st
    torch.cuda.empty_cache()
    # every sub-measurement's work, L2 flushes included, goes to the timing
    # stream, so nothing of it overlaps a timed launch
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        if not args.no_bgtq and not args.no_extras:
            line["bgtq"] = measure_bgtq(device, stream, reps=max(3, min(args.steps, 10)))
        if not args.no_extras:
            measure_extras(line, spec, device, stream)
    if rank == 0 and not args.no_cpu_baseline:
        gbs, el, sample = oracle_baseline(spec)
        cores, cpu = host_cpu()
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": cores, "cpu": cpu,
                                "kind": "oracle",
                                "sample": f"{sample}: new-token append + decode at {spec.ctx} tokens, "
                                          f"{el:.1f} s of fp64 numpy (BLAS on the process's {cores} host cores)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A case for a full ncu capture: one Qwen3-8B-shaped layer (32 q / 8 KV
    heads) at --profile-ctx tokens (default 32K; 131072 is one layer of the
    benchmark step, ~100 MB of cache), three launches of the chosen kernel:
    a decode, a fused decode step, or the append of the layer's whole
    history in one call.  decode_int2_gqa8 decodes the Llama-3-70B-shaped
    layer (64 q / 8 KV heads) at --profile-batch sequences instead."""
    torch.cuda.set_device(0)
    spec = inputs.small_spec(f"prof{args.profile_ctx // 1024}k", h_q=32, h_kv=8, batch=1, ctx=args.profile_ctx,
                             permute=True, k_kind="energy_rope", v_kind="gauss", avg_bits=3, v_bits=3, b_min=1,
                             b_max=8)
    out = torch.zeros((1, spec.h_q, spec.d), dtype=torch.float32, device="cuda")
    if args.profile_case == "append_prefill":
        # one Qwen3-8B-shaped layer's --profile-ctx history appended in one call, three times
        L = Int2Layer(spec, 0)
        k, v = L.history_kv(0)
        L.mu = inputs.key_centre(k).to("cuda").contiguous()
        sl = L.slots(0, history_positions(spec)).contiguous()
        k, v = k.contiguous(), v.contiguous()
        for _ in range(3):
            _lib.kvq_append_int2(k, v, sl, L.mu, L.R_k, L.R_v, L.cache, L.num_pages)
    elif args.profile_case == "step_int2":
        # the fused decode step (new-token append + decode) with early inputs
        L = Int2Layer(spec, 0)
        L.prefill()
        q, ws = L.queries(), L.workspace()
        k_new, v_new = L.new_kv()
        for _ in range(3):
            _lib.kvq_decode_step_int2(q, k_new, v_new, L.cache, L.num_pages, L.block_table, L.context_lens, L.mu,
                                      L.R_k, L.R_v, L.scale, out, ws, flags=_lib.KVQ_STEP_INPUTS_READY)
    elif args.profile_case in ("decode_int2", "decode_int2_gqa8"):
        if args.profile_case == "decode_int2_gqa8":
            spec = inputs.sweep70b_spec(args.profile_batch, args.profile_ctx)
            out = torch.zeros((spec.batch, spec.h_q, spec.d), dtype=torch.float32, device="cuda")
        L = Int2Layer(spec, 0)
        L.prefill()
        q, ws = L.queries(), L.workspace()
        for _ in range(3):
            _lib.kvq_decode_attn_int2(q, L.cache, L.num_pages, L.block_table, L.context_lens, L.R_k, L.R_v, L.scale,
                                      out, ws)
    else:
        L = BgtqLayer(spec, 0)
        L.prefill()
        q, ws = L.queries(), L.workspace()
        for _ in range(3):
            L.decode(q, out, ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)  # ~0.3 s timed: clock samples fall inside it
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen8b", choices=["qwen8b", "llama8b"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bgtq", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="only the headline step (e.g. for an ncu launch list)")
    ap.add_argument("--profile-case", choices=["decode_int2", "decode_int2_gqa8", "step_int2", "bgtq_decode",
                                               "append_prefill"],
                    default=None,
                    help="run a small decode case for an ncu capture instead of the benchmark")
    ap.add_argument("--profile-ctx", type=int, default=32768, help="context length of the --profile-case layer")
    ap.add_argument("--profile-batch", type=int, default=8, help="sequences of the decode_int2_gqa8 case")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
