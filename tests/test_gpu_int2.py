"""GPU parity of the INT2 path (append + fused decode) against the fp64
oracle, through the C ABI.

Bars: cache bytes (codes, fp16 scale/min) bit-exact; rotated vectors
bit-exact to the oracle's fp32 fma chain and <= 1e-5 relative to fp64;
decode outputs max |o - o_ref| <= 2e-3 * max |o_ref|.
"""
import math

import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer, history_positions
from oracle import int2

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _f64(x):
    return x.detach().cpu().to(torch.float64).numpy()


def _np_f32(x):
    return x.detach().cpu().to(torch.float32).numpy()


def _close(got, want, tol=TOL):
    err = np.max(np.abs(got - want))
    ref = np.max(np.abs(want))
    assert np.all(np.isfinite(got))
    assert err <= tol * ref, f"max err {err:.3e} vs {tol} * {ref:.3e}"
    return err / ref


def _append_all(layer: Int2Layer, with_dbg=False):
    """GPU: prefill every sequence, then the decode token (two calls)."""
    spec = layer.spec
    pos = history_positions(spec)
    ks, vs, sls = [], [], []
    for b in range(spec.batch):
        k, v = layer.history_kv(b, device="cpu")
        ks.append(k)
        vs.append(v)
        sls.append(inputs.slot_mapping(layer.block_table[b].cpu(), pos))
    k_new, v_new = layer.new_kv(device="cpu")
    k_all = torch.cat(ks + [k_new])
    v_all = torch.cat(vs + [v_new])
    sl_all = torch.cat(sls + [torch.cat([inputs.slot_mapping(layer.block_table[b].cpu(), torch.tensor([spec.ctx - 1]))
                                         for b in range(spec.batch)])])
    layer.mu = inputs.key_centre(ks[0]).to(layer.device)
    dev = layer.device
    n_hist = sum(k.shape[0] for k in ks)
    dbg_k = torch.zeros((k_all.shape[0], spec.h_kv, 128), dtype=torch.float32, device=dev) if with_dbg else None
    dbg_v = torch.zeros_like(dbg_k) if with_dbg else None
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kd, vd, sd = k_all.to(dev), v_all.to(dev), sl_all.to(dev)
    _lib.kvq_append_int2(kd[:n_hist], vd[:n_hist], sd[:n_hist], layer.mu, layer.R_k, layer.R_v, layer.cache,
                         layer.num_pages, None if dbg_k is None else dbg_k[:n_hist],
                         None if dbg_v is None else dbg_v[:n_hist], err)
    _lib.kvq_append_int2(kd[n_hist:], vd[n_hist:], sd[n_hist:], layer.mu, layer.R_k, layer.R_v, layer.cache,
                         layer.num_pages, None if dbg_k is None else dbg_k[n_hist:],
                         None if dbg_v is None else dbg_v[n_hist:], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return k_all, v_all, sl_all, dbg_k, dbg_v


def _oracle_cache(layer: Int2Layer, k_all, v_all, sl_all, exact=True):
    cache = int2.new_cache(layer.num_pages, layer.spec.h_kv)
    info = int2.append(cache, _np_f32(k_all), _np_f32(v_all), sl_all.numpy(), _np_f32(layer.mu),
                       _np_f32(layer.R_k), _np_f32(layer.R_v), exact_chain=exact)
    return cache, info


def _decode_gpu(layer: Int2Layer, q, num_splits=0, context_lens=None):
    spec = layer.spec
    out = torch.full((spec.batch, spec.h_q, 128), float("nan"), dtype=torch.float32, device=layer.device)
    ws = layer.workspace(num_splits)
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table,
                              layer.context_lens if context_lens is None else context_lens,
                              layer.R_k, layer.R_v, layer.scale, out, ws, num_splits)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    assert int(ws[256:256 + 4 * spec.batch * spec.h_kv].view(torch.int32).abs().sum()) == 0  # tickets reset
    return out


# --------------------------------------------------------------------------- append

def test_append_bit_exact_tiny():
    spec = inputs.SPECS["tiny"]
    layer = Int2Layer(spec, 0)
    k_all, v_all, sl_all, dbg_k, dbg_v = _append_all(layer, with_dbg=True)
    cache, info = _oracle_cache(layer, k_all, v_all, sl_all)
    # rotated vectors: bit-exact to the fp32 fma chain, <= 1e-5 relative to fp64
    assert np.array_equal(_np_f32(dbg_k), info["z"])
    assert np.array_equal(_np_f32(dbg_v), info["w"])
    for h in range(spec.h_kv):
        _, z64 = int2.rotate_keys(_np_f32(k_all[:, h]), _np_f32(layer.mu[h]), _np_f32(layer.R_k[h]), False)
        rel = np.max(np.abs(_np_f32(dbg_k[:, h]) - z64), axis=1) / np.max(np.abs(z64), axis=1)
        assert rel.max() <= 1e-5
    assert np.array_equal(layer.cache.cpu().numpy(), cache)


def test_append_adversarial_bit_exact():
    """Exact level values and midpoints, constant groups, fp16 overflow and
    underflow of scale/min, skipped (-1) and out-of-range slots."""
    torch.manual_seed(0)
    spec = inputs.small_spec("adv", ctx=64)
    layer = Int2Layer(spec, 0, block_table=torch.tensor([[3, 1, 0, 2]], dtype=torch.int32))
    eye = torch.eye(128, dtype=torch.float32, device="cuda")[None].contiguous()
    layer.R_k, layer.R_v = eye, eye.clone()
    n = 48
    k = torch.randn(n, 1, 128) * 3
    k[0, 0, :32] = 1.5                                   # constant group
    k[1, 0, :32] = torch.tensor([0.0, 3.0] + [0.5, 1.0, 1.5, 2.0, 2.5] * 6)  # exact midpoints
    k[2, 0, 32:64] = 1e5 * torch.sign(torch.randn(32))   # fp16 overflow -> saturate
    k[3, 0, 64:96] = 1e-8 * torch.randn(32)              # scale underflow
    k[4, 0, 96:] = torch.linspace(-1, 1, 32)
    v = torch.randn(n, 1, 128)
    v[5, 0, :64] = -7.25
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    slots = torch.arange(n, dtype=torch.int32) + 16
    slots[7] = -1
    slots[9] = 64 * 16                                   # beyond the pool: skipped and counted
    mu = torch.zeros(1, 128, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.cache.fill_(0)
    _lib.kvq_append_int2(k.cuda(), v.cuda(), slots.cuda(), mu, layer.R_k, layer.R_v, layer.cache, layer.num_pages,
                         None, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    cache = int2.new_cache(layer.num_pages, 1)
    sl = slots.numpy().copy()
    sl[9] = -1
    int2.append(cache, _np_f32(k), _np_f32(v), sl, np.zeros((1, 128), np.float32), np.eye(128, dtype=np.float32)[None],
                np.eye(128, dtype=np.float32)[None])
    assert np.array_equal(layer.cache.cpu().numpy(), cache)


@pytest.mark.parametrize("clip", [1.0, 0.9])
def test_prefill_append_matches_token_appends_and_oracle(clip):
    """A 1000-token append takes the register-tiled prefill kernel: its cache
    bytes, rotated vectors and error count equal those of the same tokens
    appended 200 at a time (the per-token kernel) and the oracle's cache."""
    torch.manual_seed(3)
    h_kv, n = 2, 1000
    spec = inputs.small_spec("pfapp", h_q=8, h_kv=h_kv, ctx=1024)
    layer = Int2Layer(spec, 0)
    k = (torch.randn(n, h_kv, 128) * 2 + torch.randn(1, h_kv, 128) * 3).to(torch.bfloat16)
    v = torch.randn(n, h_kv, 128).to(torch.bfloat16)
    k[10, 0, :32] = 1.5                                   # constant group
    bt = layer.block_table[0].cpu()
    slots = inputs.slot_mapping(bt, torch.arange(n)).to(torch.int32)
    slots[17] = -1
    slots[500] = -1
    slots[333] = layer.num_pages * 16 + 5                 # beyond the pool: skipped and counted
    slots[999] = -7                                       # invalid: skipped and counted
    mu = inputs.key_centre(k).to("cuda").contiguous()
    kd, vd, sd = k.cuda().contiguous(), v.cuda().contiguous(), slots.cuda().contiguous()
    outs = []
    for step in (n, 200):
        layer.cache.fill_(0)
        dk = torch.zeros((n, h_kv, 128), dtype=torch.float32, device="cuda")
        dv = torch.zeros_like(dk)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for t0 in range(0, n, step):
            t1 = min(n, t0 + step)
            _lib.kvq_append_int2_clip(kd[t0:t1], vd[t0:t1], sd[t0:t1], mu, layer.R_k, layer.R_v, clip, layer.cache,
                                      layer.num_pages, dk[t0:t1], dv[t0:t1], err)
        torch.cuda.synchronize()
        outs.append((layer.cache.cpu().numpy().copy(), _np_f32(dk), _np_f32(dv), int(err.item())))
    (c_big, dk_big, dv_big, e_big), (c_small, dk_small, dv_small, e_small) = outs
    assert e_big == e_small == 2
    assert np.array_equal(c_big, c_small)
    assert np.array_equal(dk_big, dk_small) and np.array_equal(dv_big, dv_small)
    sl = slots.numpy().copy()
    sl[333] = sl[999] = -1
    cache = int2.new_cache(layer.num_pages, h_kv)
    info = int2.append(cache, _np_f32(k), _np_f32(v), sl, _np_f32(mu), _np_f32(layer.R_k), _np_f32(layer.R_v),
                       clip=clip)
    assert np.array_equal(c_big, cache)
    keep = sl >= 0
    assert np.array_equal(dk_big[keep], info["z"][keep]) and np.array_equal(dv_big[keep], info["w"][keep])


def test_prefill_append_unaligned_inputs_take_the_token_kernel():
    """Inputs that are not 16-byte aligned go to the per-token kernel; the
    cache comes out the same as from aligned inputs."""
    torch.manual_seed(5)
    h_kv, n = 2, 600
    spec = inputs.small_spec("pfal", h_q=8, h_kv=h_kv, ctx=640)
    layer = Int2Layer(spec, 0)
    k = torch.randn(n, h_kv, 128).to(torch.bfloat16).cuda()
    v = torch.randn(n, h_kv, 128).to(torch.bfloat16).cuda()
    slots = inputs.slot_mapping(layer.block_table[0].cpu(), torch.arange(n)).to(torch.int32).cuda()
    mu = torch.zeros(h_kv, 128, device="cuda")
    caches = []
    for shift in (0, 4):  # 4 bf16 = 8 bytes: 8-byte but not 16-byte aligned
        bk = torch.empty(n * h_kv * 128 + shift, dtype=torch.bfloat16, device="cuda")
        bv = torch.empty_like(bk)
        kk, vv = bk[shift:].view(n, h_kv, 128), bv[shift:].view(n, h_kv, 128)
        kk.copy_(k)
        vv.copy_(v)
        assert (kk.data_ptr() % 16 == 0) == (shift == 0)
        layer.cache.fill_(0)
        _lib.kvq_append_int2(kk, vv, slots, mu, layer.R_k, layer.R_v, layer.cache, layer.num_pages)
        torch.cuda.synchronize()
        caches.append(layer.cache.cpu().numpy().copy())
    assert np.array_equal(caches[0], caches[1])


# --------------------------------------------------------------------------- decode

def test_decode_tiny_end_to_end():
    spec = inputs.SPECS["tiny"]
    layer = Int2Layer(spec, 0)
    k_all, v_all, sl_all, _, _ = _append_all(layer)
    cache, _ = _oracle_cache(layer, k_all, v_all, sl_all)
    assert np.array_equal(layer.cache.cpu().numpy(), cache)
    q = layer.queries()
    ref = int2.decode(_f64(q), cache, layer.block_table.cpu().numpy(), [spec.ctx] * spec.batch, _np_f32(layer.mu),
                      _np_f32(layer.R_k), _np_f32(layer.R_v), layer.scale, spec.h_kv)
    for splits in (0, 1, 3, 40):
        _close(_decode_gpu(layer, q, splits).cpu().numpy(), ref)


@pytest.mark.parametrize("h_q,h_kv,ctxs,splits,permute", [
    (4, 1, [1], 0, False),
    (4, 2, [17, 300], 0, True),
    (8, 8, [33, 1000, 5, 16], 0, True),          # GQA 1
    (16, 8, [250, 64], 4, True),                  # GQA 2
    (24, 8, [129], 2, True),                      # GQA 3
    (64, 8, [700, 1500], 0, True),                # GQA 8
    (32, 4, [2049, 3, 511], 7, True),             # ragged, GQA 8
    (8, 2, [40], 64, False),                      # more splits than pages
])
def test_decode_shapes_on_oracle_cache(h_q, h_kv, ctxs, splits, permute):
    """Decode over a cache the oracle wrote (uploaded), ragged lengths,
    several splits, GQA groups 1..8."""
    B = len(ctxs)
    spec = inputs.small_spec(f"shape{h_q}_{h_kv}_{B}", h_q=h_q, h_kv=h_kv, batch=B, ctx=max(ctxs), permute=permute)
    layer = Int2Layer(spec, 0, extra_pages=3)
    rng = np.random.default_rng(h_q * 7 + B)
    ctx_lens = np.array(ctxs, dtype=np.int32)
    cache = int2.new_cache(layer.num_pages, h_kv)
    mu = (rng.standard_normal((h_kv, 128)) * 2).astype(np.float32)
    layer.mu = torch.as_tensor(mu, device="cuda")
    bt = layer.block_table.cpu().numpy()
    for b in range(B):
        T = int(ctx_lens[b])
        k = (rng.standard_normal((T, h_kv, 128)) * 2 + rng.standard_normal(128) * 3).astype(np.float32)
        v = rng.standard_normal((T, h_kv, 128)).astype(np.float32)
        k = torch.as_tensor(k).to(torch.bfloat16).float().numpy()
        v = torch.as_tensor(v).to(torch.bfloat16).float().numpy()
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        int2.append(cache, k, v, slots, mu, _np_f32(layer.R_k), _np_f32(layer.R_v), exact_chain=False)
    # stale garbage (including NaN scales) in the unused slots of the last pages
    cache_gpu = cache.copy()
    for b in range(B):
        T = int(ctx_lens[b])
        if T % 16:
            tile = cache_gpu[bt[b, (T - 1) // 16]]
            for s in range(T % 16, 16):
                tile[:, int2.meta_bytes(0, s)] = 0xFF
                tile[:, int2.meta_bytes(1, s)] = 0xFF
                tile[:, int2.OFF_V_CODES + 32 * s: int2.OFF_V_CODES + 32 * s + 32] = 0xFF
    layer.cache.copy_(torch.as_tensor(cache_gpu))
    cl = torch.as_tensor(ctx_lens, device="cuda")
    q = torch.as_tensor(rng.standard_normal((B, h_q, 128)), dtype=torch.bfloat16).cuda()
    ref = int2.decode(_f64(q), cache, bt, ctx_lens, mu, _np_f32(layer.R_k), _np_f32(layer.R_v), layer.scale, h_kv)
    got = _decode_gpu(layer, q, splits, context_lens=cl).cpu().numpy()
    for b in range(B):
        _close(got[b], ref[b])


def test_decode_empty_context_and_bad_page():
    spec = inputs.small_spec("edge", h_q=4, h_kv=1, batch=3, ctx=40)
    layer = Int2Layer(spec, 0)
    layer.mu = torch.zeros(1, 128, device="cuda")
    q = torch.randn(3, 4, 128).to(torch.bfloat16).cuda()
    cl = torch.tensor([0, 40, 20], dtype=torch.int32, device="cuda")
    out = _decode_gpu(layer, q, 0, context_lens=cl).cpu()
    assert torch.all(out[0] == 0)
    assert torch.isfinite(out).all()
    bt = layer.block_table.clone()
    bt[1, 1] = layer.num_pages + 5
    layer.block_table = bt
    ws = layer.workspace()
    out = torch.zeros(3, 4, 128, device="cuda")
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, cl, layer.R_k, layer.R_v,
                              layer.scale, out, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == -5
    assert _lib.kvq_workspace_status(ws) == 0
    assert torch.isfinite(out).all()


def test_decode_rejects_small_workspace():
    spec = inputs.small_spec("ws", h_q=4, h_kv=1, batch=1, ctx=40)
    layer = Int2Layer(spec, 0)
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 4, 128, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.KvqError) as e:
        _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens, layer.R_k,
                                  layer.R_v, layer.scale, out, ws)
    assert e.value.status == -3


# --------------------------------------------------------------------------- full-size sampled

def _sampled_check(spec, layer_idx, samples, splits=0, token_samples=256, exact=False):
    layer = Int2Layer(spec, layer_idx)
    layer.prefill()
    k_new, v_new = layer.new_kv()
    _lib.kvq_append_int2(k_new, v_new, layer.new_slots(), layer.mu, layer.R_k, layer.R_v, layer.cache,
                         layer.num_pages)
    q = layer.queries()
    got = _decode_gpu(layer, q, splits).cpu().numpy()
    bt = layer.block_table.cpu().numpy()
    rng = np.random.default_rng(layer_idx)
    mu = _np_f32(layer.mu)
    for b, h in samples:
        k, v = layer.history_kv(b)
        k = torch.cat([k, k_new[b:b + 1]])[:, h:h + 1]
        v = torch.cat([v, v_new[b:b + 1]])[:, h:h + 1]
        T = spec.ctx
        kf, vf = _np_f32(k), _np_f32(v)
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        rk, rv = _np_f32(layer.R_k[h:h + 1]), _np_f32(layer.R_v[h:h + 1])
        # codes of sampled tokens: bit-exact against the fp32 chain
        idx = np.sort(rng.choice(T, size=min(token_samples, T), replace=False))
        small = int2.new_cache(layer.num_pages, 1)
        int2.append(small, kf[idx], vf[idx], slots[idx], mu[h:h + 1], rk, rv, exact_chain=True)
        gpu_tiles = layer.cache[:, h].cpu().numpy()
        for t in idx:
            page, s = divmod(int(slots[t]), 16)
            for idx in (int2.OFF_K_CODES + 32 * s + np.arange(32), int2.meta_bytes(0, s),
                        int2.OFF_V_CODES + 32 * s + np.arange(32), int2.meta_bytes(1, s)):
                assert np.array_equal(gpu_tiles[page, idx], small[page, 0, idx]), (b, h, t)
        # attention of the sampled (sequence, KV head); with exact=False the
        # oracle decides codes from its fp64 rotation (rare ties differ)
        full = int2.new_cache(layer.num_pages, 1)
        int2.append(full, kf, vf, slots, mu[h:h + 1], rk, rv, exact_chain=exact)
        g = spec.g
        ref = int2.decode(_f64(q[b:b + 1, h * g:(h + 1) * g]), full, bt[b:b + 1], [T], mu[h:h + 1], rk, rv,
                          layer.scale, 1)
        _close(got[b, h * g:(h + 1) * g], ref[0])


def test_llama8b_full_size_sampled():
    # post-RoPE keys with heavy offsets give peaked attention, where one
    # flipped code of a dominant token shows: decide codes exactly
    _sampled_check(inputs.SPECS["llama8b"], 0, [(0, 0), (7, 7)], exact=True)


def test_qwen8b_full_context_sampled_layers():
    spec = inputs.SPECS["qwen8b"]
    _sampled_check(spec, 0, [(0, 2)])
    _sampled_check(spec, 35, [(0, 6)])


# The 70B-class GQA-8 scaling grid: batch {1, 8, 32, 64} x context {4K, 32K,
# 128K}, and batch 1 at 256K and 512K.  Each point is decoded in full on the
# GPU (automatic split) and checked on sampled (sequence, KV head) pairs.
SWEEP = [(B, T) for B in (1, 8, 32, 64) for T in (4096, 32768, 131072)] + [(1, 262144), (1, 524288)]


@pytest.mark.parametrize("B,T", SWEEP, ids=[f"b{B}_t{T // 1024}k" for B, T in SWEEP])
def test_sweep70b_point_sampled(B, T):
    rng = np.random.default_rng(B * 7 + T)
    samples = sorted({(int(rng.integers(0, B)), int(rng.integers(0, 8))) for _ in range(2 if T <= 32768 else 1)})
    if B > 1:
        samples.append((B - 1, 7))                  # the last unit of the page split
    _sampled_check(inputs.sweep70b_spec(B, T), 0, samples, token_samples=64 if T > 4096 else 128)


def test_sweep70b_batch64_explicit_split():
    # 64 sequences x 8 KV heads at one CTA each: a grid of 3.4 waves of 152
    _sampled_check(inputs.sweep70b_spec(64, 4096), 0, [(0, 0), (37, 5), (63, 7)], splits=1, token_samples=64)
