"""GPU parity of the INT2 decode with a BF16 window (sink / recent tokens
kept unquantised) against the fp64 oracle, through the C ABI.

"Output-Aware Rotation for INT2 KV-Cache Quantization" §3.1 keeps a small
BF16 window; the Block-GTQ page keeps 4 sink + 128 recent tokens (Table 6).
Bar: max |o - o_ref| <= 2e-3 * max |o_ref| per sequence, as for the plain
decode.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer
from oracle import int2

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _np_f32(x):
    return x.detach().cpu().to(torch.float32).numpy()


def _bf16_round(a):
    return torch.as_tensor(a).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("h_q,h_kv,ctxs,wins,win_max,splits", [
    (32, 8, [300, 1000], [132, 0], 132, 0),      # GQA 4: 4 sinks + 128 recent, and no window
    (64, 8, [700], [37], 64, 3),                  # GQA 8, explicit splits
    (8, 2, [0, 50], [5, 1], 8, 0),                # window only; a one-token window
    (4, 1, [17], [128], 128, 2),                  # window longer than the cached part
    (16, 4, [2049, 33, 160], [1, 132, 200], 200, 7),  # ragged, a full window
    # from 96 pages up a unit's share carries window pages without work: the
    # automatic split (shares crossing unit ends, the window attended by the
    # CTA holding a unit's last virtual page) and one CTA per unit
    (32, 8, [3000, 1600], [132, 60], 132, 0),
    (32, 8, [2000], [132], 132, 1),
    (8, 2, [2000, 1700], [700, 333], 700, 0),    # window past the 256-page balance cap
])
def test_window_decode_matches_oracle(h_q, h_kv, ctxs, wins, win_max, splits):
    B = len(ctxs)
    spec = inputs.small_spec(f"win{h_q}_{h_kv}_{B}", h_q=h_q, h_kv=h_kv, batch=B, ctx=max(max(ctxs), 16),
                             permute=True)
    layer = Int2Layer(spec, 0, extra_pages=2)
    rng = np.random.default_rng(h_q * 13 + B + win_max)
    ctx_lens = np.array(ctxs, dtype=np.int32)
    mu = (rng.standard_normal((h_kv, 128)) * 2).astype(np.float32)
    bt = layer.block_table.cpu().numpy()
    cache = int2.new_cache(layer.num_pages, h_kv)
    for b in range(B):
        T = int(ctx_lens[b])
        if T == 0:
            continue
        k = _bf16_round((rng.standard_normal((T, h_kv, 128)) * 2 + rng.standard_normal(128) * 3).astype(np.float32))
        v = _bf16_round(rng.standard_normal((T, h_kv, 128)).astype(np.float32))
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        int2.append(cache, k, v, slots, mu, _np_f32(layer.R_k), _np_f32(layer.R_v), exact_chain=False)
    cache_gpu = cache.copy()
    for b in range(B):                       # stale bytes (NaN scales) past each context
        T = int(ctx_lens[b])
        if T % 16:
            tile = cache_gpu[bt[b, (T - 1) // 16]]
            for s in range(T % 16, 16):
                tile[:, int2.meta_bytes(0, s)] = 0xFF
                tile[:, int2.meta_bytes(1, s)] = 0xFF
    layer.cache.copy_(torch.as_tensor(cache_gpu))
    kw = _bf16_round((rng.standard_normal((B, win_max, h_kv, 128)) * 2 + mu * 0.5).astype(np.float32))
    vw = _bf16_round(rng.standard_normal((B, win_max, h_kv, 128)).astype(np.float32))
    lens = np.array(wins, dtype=np.int32)
    q = torch.as_tensor(rng.standard_normal((B, h_q, 128)), dtype=torch.bfloat16).cuda()
    ref = int2.decode(q.cpu().double().numpy(), cache, bt, ctx_lens, mu, _np_f32(layer.R_k), _np_f32(layer.R_v),
                      layer.scale, h_kv, window=(kw, vw, lens))
    nbytes = _lib.kvq_decode_workspace_bytes(B, h_q, h_kv, bt.shape[1], splits + 1 if splits else 0)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((B, h_q, 128), float("nan"), device="cuda")
    _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table,
                                     torch.as_tensor(ctx_lens, device="cuda"), layer.R_k, layer.R_v,
                                     torch.as_tensor(mu, device="cuda"),
                                     torch.as_tensor(kw, dtype=torch.bfloat16, device="cuda"),
                                     torch.as_tensor(vw, dtype=torch.bfloat16, device="cuda"),
                                     torch.as_tensor(lens, device="cuda"), layer.scale, out, ws, splits)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    assert int(ws[256:256 + 4 * B * h_kv].view(torch.int32).abs().sum()) == 0   # tickets reset
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in range(B):
        err = np.max(np.abs(got[b] - ref[b]))
        assert err <= TOL * np.max(np.abs(ref[b])), (b, err, np.max(np.abs(ref[b])))


def test_window_zero_lengths_match_plain_decode():
    # win_lens all zero: the window split contributes nothing, so the result
    # matches kvq_decode_attn_int2 on the same cache to fp32 rounding.
    spec = inputs.small_spec("winzero", h_q=32, h_kv=8, batch=2, ctx=900, permute=True)
    layer = Int2Layer(spec, 0)
    layer.prefill()
    q = layer.queries()
    ws = layer.workspace()
    plain = torch.zeros((2, 32, 128), device="cuda")
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens, layer.R_k,
                              layer.R_v, layer.scale, plain, ws)
    kw = torch.randn(2, 4, 8, 128, device="cuda").to(torch.bfloat16)
    win = torch.zeros((2, 32, 128), device="cuda")
    _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                     layer.R_k, layer.R_v, layer.mu, kw, kw, torch.zeros(2, dtype=torch.int32,
                                                                                         device="cuda"),
                                     layer.scale, win, ws)
    torch.cuda.synchronize()
    err = (win - plain).abs().max().item()
    assert err <= 1e-5 * plain.abs().max().item()


def test_sole_partial_output_equals_its_merge_bit_for_bit():
    # one split per unit: the plain decode's CTA is each unit's only partial
    # and writes the output directly; the window form adds an (empty) window
    # partial, so the same page partial goes through the slot, ticket and
    # merge.  Merging one partial with an empty one is exact, so the two
    # outputs must be identical.
    spec = inputs.small_spec("solepart", h_q=16, h_kv=4, batch=3, ctx=700, permute=True)
    layer = Int2Layer(spec, 0)
    layer.prefill()
    q = layer.queries()
    ws = layer.workspace(2)
    plain = torch.full((3, 16, 128), float("nan"), device="cuda")
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens, layer.R_k,
                              layer.R_v, layer.scale, plain, ws, 1)
    kw = torch.randn(3, 4, 4, 128, device="cuda").to(torch.bfloat16)
    win = torch.full((3, 16, 128), float("nan"), device="cuda")
    _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                     layer.R_k, layer.R_v, layer.mu, kw, kw,
                                     torch.zeros(3, dtype=torch.int32, device="cuda"), layer.scale, win, ws, 1)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    assert torch.isfinite(plain).all()
    assert torch.equal(plain, win)


def test_window_argument_checks():
    spec = inputs.small_spec("winarg", h_q=4, h_kv=1, batch=1, ctx=40)
    layer = Int2Layer(spec, 0)
    layer.mu = torch.zeros(1, 128, device="cuda")
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 4, 128, device="cuda")
    kw = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(_lib.kvq_decode_workspace_bytes(1, 4, 1, layer.block_table.shape[1], 1), dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(_lib.KvqError) as e:    # 1 unit + 2 page CTAs + the window partial need 4 slots, 3 are there
        _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                         layer.R_k, layer.R_v, layer.mu, kw, kw, lens, layer.scale, out, small, 2)
    assert e.value.status == -3


def test_qwen8b_window_full_size_sampled():
    """The timed window workload: one Qwen3-8B-shaped layer at 128K (the
    decode token appended) and a window of 4 sink + 128 recent tokens per
    sequence, decoded in full with the automatic split; the first and the
    last KV head (whose shares hold the ends of the page space) are checked
    against the oracle."""
    spec = inputs.SPECS["qwen8b"]
    layer = Int2Layer(spec, 0)
    layer.prefill()
    k_new, v_new = layer.new_kv()
    _lib.kvq_append_int2(k_new, v_new, layer.new_slots(), layer.mu, layer.R_k, layer.R_v, layer.cache,
                         layer.num_pages)
    q = layer.queries()
    w = inputs.WINDOW_SINK + inputs.WINDOW_RECENT
    rng = np.random.default_rng(132)
    mu = _np_f32(layer.mu)
    kw = _bf16_round((rng.standard_normal((spec.batch, w, spec.h_kv, 128)) * 2 + mu * 0.5).astype(np.float32))
    vw = _bf16_round(rng.standard_normal((spec.batch, w, spec.h_kv, 128)).astype(np.float32))
    lens = np.full(spec.batch, w, dtype=np.int32)
    out = torch.full((spec.batch, spec.h_q, 128), float("nan"), device="cuda")
    ws = layer.workspace()
    _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                     layer.R_k, layer.R_v, layer.mu,
                                     torch.as_tensor(kw, dtype=torch.bfloat16, device="cuda"),
                                     torch.as_tensor(vw, dtype=torch.bfloat16, device="cuda"),
                                     torch.as_tensor(lens, device="cuda"), layer.scale, out, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    bt = layer.block_table.cpu().numpy()
    T, g = spec.ctx, spec.g
    for b, h in [(0, 0), (spec.batch - 1, spec.h_kv - 1)]:
        k, v = layer.history_kv(b)
        kf = _np_f32(torch.cat([k, k_new[b:b + 1]])[:, h:h + 1])
        vf = _np_f32(torch.cat([v, v_new[b:b + 1]])[:, h:h + 1])
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        rk, rv = _np_f32(layer.R_k[h:h + 1]), _np_f32(layer.R_v[h:h + 1])
        full = int2.new_cache(layer.num_pages, 1)
        int2.append(full, kf, vf, slots, mu[h:h + 1], rk, rv, exact_chain=False)
        ref = int2.decode(q[b:b + 1, h * g:(h + 1) * g].cpu().double().numpy(), full, bt[b:b + 1], [T],
                          mu[h:h + 1], rk, rv, layer.scale, 1,
                          window=(kw[b:b + 1, :, h:h + 1], vw[b:b + 1, :, h:h + 1], lens[b:b + 1]))
        err = np.max(np.abs(got[b, h * g:(h + 1) * g] - ref[0]))
        assert err <= TOL * np.max(np.abs(ref[0])), (b, h, err, np.max(np.abs(ref[0])))
