"""GPU parity of the fused decode step (kvq_decode_step_int2): the new
token's cache bytes equal kvq_append_int2's bit for bit, and the attention
over the context, new token included, matches the fp64 oracle within
2e-3 * max|o_ref| (and the two-call path up to the merge's rounding order).

Output-Aware Rotation for INT2 KV-Cache Quantization: §1 and §3.1 Eq. (4)
(quantise-on-append of the rotated, centred key and the rotated value), §3
Eqs. (1)-(2) (attention over s <= t, the new token included).
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer
from oracle import int2

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _np(x):
    return x.detach().cpu().to(torch.float32).numpy()


@pytest.mark.parametrize("h_q,h_kv,ctxs,splits", [
    (32, 8, [1000, 1025], 0),        # the new token at slot 7 of a page / first slot of a new page
    (8, 2, [1, 16, 17, 300], 0),     # only the new token; the last slot of a page; ragged
    (64, 8, [700, 33], 0),           # GQA 8
    (12, 4, [2048, 0, 5], 3),        # GQA 3, an empty sequence, explicit splits
])
def test_step_matches_append_then_decode_and_oracle(h_q, h_kv, ctxs, splits):
    B = len(ctxs)
    spec = inputs.small_spec(f"step{h_q}{h_kv}{B}", h_q=h_q, h_kv=h_kv, batch=B, ctx=max(max(ctxs), 1), permute=True)
    a = Int2Layer(spec, 0, extra_pages=1)
    # history of every sequence (ctx - 1 tokens) through the append kernel
    k0, _ = a.history_kv(0)
    a.mu = inputs.key_centre(k0).cuda().contiguous()
    hist = []
    for b, T in enumerate(ctxs):
        k, v = a.history_kv(b)
        n = max(T - 1, 0)
        k, v = k[:n].contiguous(), v[:n].contiguous()
        hist.append((k, v))
        if n:
            _lib.kvq_append_int2(k, v, a.slots(b, torch.arange(n)), a.mu, a.R_k, a.R_v, a.cache, a.num_pages)
    cl = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    k_new, v_new = a.new_kv()
    q = a.queries()
    # two calls: append of the new tokens, then decode
    b2 = Int2Layer(spec, 0, extra_pages=1)
    b2.mu = a.mu
    b2.cache.copy_(a.cache)
    rows = [b for b, T in enumerate(ctxs) if T > 0]
    slots = torch.cat([a.slots(b, torch.tensor([ctxs[b] - 1])) for b in rows])
    _lib.kvq_append_int2(k_new[rows].contiguous(), v_new[rows].contiguous(), slots, b2.mu, b2.R_k, b2.R_v, b2.cache,
                         b2.num_pages)
    ws2 = b2.workspace(splits)
    two = torch.zeros((B, h_q, 128), device="cuda")
    _lib.kvq_decode_attn_int2(q, b2.cache, b2.num_pages, b2.block_table, cl, b2.R_k, b2.R_v, b2.scale, two, ws2,
                              splits)
    # one launch, with the inputs read after the dependency wait, then (on a
    # copy of the starting cache) with the early-inputs flag: the same bytes
    # and the same output
    start = a.cache.clone()
    ws = a.workspace(splits)
    out_ready = torch.full((B, h_q, 128), float("nan"), device="cuda")
    _lib.kvq_decode_step_int2(q, k_new, v_new, a.cache, a.num_pages, a.block_table, cl, a.mu, a.R_k, a.R_v, a.scale,
                              out_ready, ws, splits, flags=_lib.KVQ_STEP_INPUTS_READY)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    ready_cache = a.cache.clone()
    a.cache.copy_(start)
    out = torch.full((B, h_q, 128), float("nan"), device="cuda")
    _lib.kvq_decode_step_int2(q, k_new, v_new, a.cache, a.num_pages, a.block_table, cl, a.mu, a.R_k, a.R_v, a.scale,
                              out, ws, splits)
    torch.cuda.synchronize()
    assert torch.equal(a.cache, ready_cache) and torch.equal(out, out_ready)
    assert _lib.kvq_workspace_status(ws) == 0
    assert int(ws[256:256 + 4 * B * h_kv].view(torch.int32).abs().sum()) == 0   # tickets reset
    assert torch.equal(a.cache, b2.cache)                                       # the same bytes as the append
    got, want2 = out.cpu().numpy(), two.cpu().numpy()
    assert np.all(np.isfinite(got))
    # the oracle: its own cache from the same tokens, decode in fp64
    cache = int2.new_cache(a.num_pages, h_kv)
    bt = a.block_table.cpu().numpy()
    mu, rk, rv = _np(a.mu), _np(a.R_k), _np(a.R_v)
    for b, T in enumerate(ctxs):
        if T == 0:
            continue
        k, v = hist[b]
        kk = torch.cat([k.cpu(), k_new[b:b + 1].cpu()])
        vv = torch.cat([v.cpu(), v_new[b:b + 1].cpu()])
        sl = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        int2.append(cache, _np(kk), _np(vv), sl, mu, rk, rv)
    assert np.array_equal(a.cache.cpu().numpy(), cache)
    ref = int2.decode(q.cpu().double().numpy(), cache, bt, ctxs, mu, rk, rv, a.scale, h_kv)
    for b, T in enumerate(ctxs):
        if T == 0:
            assert np.all(got[b] == 0)
            continue
        scale = np.max(np.abs(ref[b]))
        assert np.max(np.abs(got[b] - ref[b])) <= TOL * scale
        assert np.max(np.abs(got[b] - want2[b])) <= 1e-4 * scale


def test_step_bad_page_of_the_new_token_is_reported():
    spec = inputs.small_spec("stepbad", h_q=4, h_kv=1, batch=1, ctx=40)
    a = Int2Layer(spec, 0)
    a.prefill()
    bt = a.block_table.clone()
    bt[0, 2] = a.num_pages + 5                    # the page of position 39
    k_new, v_new = a.new_kv()
    out = torch.zeros((1, 4, 128), device="cuda")
    ws = a.workspace()
    before = a.cache.clone()
    _lib.kvq_decode_step_int2(a.queries(), k_new, v_new, a.cache, a.num_pages, bt, a.context_lens, a.mu, a.R_k,
                              a.R_v, a.scale, out, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == -5
    assert torch.equal(a.cache, before)
    assert torch.isfinite(out).all()
