"""GPU parity of the Block-GTQ path (grouped TQ-MSE append + fused decode)
against the fp64 oracle, through the C ABI.

Bars: cache bytes (bit streams, fp16 norms) bit-exact; decode outputs
max |o - o_ref| <= 2e-3 * max |o_ref|.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import BgtqLayer, history_positions
from oracle import attention, bgtq

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def table():
    return bgtq.lloyd_max_table()


def _f32(x):
    return x.detach().cpu().float().numpy()


def _close(got, want, tol=TOL):
    err = np.max(np.abs(got - want))
    ref = np.max(np.abs(want))
    assert np.all(np.isfinite(got))
    assert err <= tol * ref, f"max err {err:.3e} vs {tol} * {ref:.3e}"


def _pis(layer):
    return bgtq.tq_rotation_dict(layer.pi_table64, layer.pi_offsets_np)


def _spec(name, **kw):
    base = dict(h_q=8, h_kv=2, batch=1, ctx=100, k_kind="energy_rope", v_kind="gauss", avg_bits=3, v_bits=3,
                b_min=1, b_max=8)
    base.update(kw)
    return inputs.small_spec(name, **base)


def _append_both(layer, table, k, v, slots):
    layer.append(k.cuda().contiguous(), v.cuda().contiguous(), slots.cuda().contiguous())
    torch.cuda.synchronize()
    cache = bgtq.new_cache(layer.num_pages, layer.spec.h_kv, layer.total_bits, layer.v_bits)
    bgtq.append(cache, _f32(k), _f32(v), slots.numpy(), layer.widths_np, layer.v_bits, layer.total_bits, _pis(layer),
                table)
    return cache


@pytest.mark.parametrize("avg_bits,v_bits,b_max", [(3, 3, 8), (2, 2, 8), (1, 1, 8), (8, 8, 8), (4, 5, 6)])
def test_append_bit_exact(table, avg_bits, v_bits, b_max):
    spec = _spec(f"bgapp{avg_bits}{v_bits}", ctx=40, avg_bits=avg_bits, v_bits=v_bits, b_max=b_max)
    layer = BgtqLayer(spec, 0, codebooks=table)
    k, v = layer.history_kv(0, device="cpu")
    k[3] = 0                                      # zero key and value vectors
    v[5] = 0
    slots = inputs.slot_mapping(layer.block_table[0].cpu(), history_positions(spec))
    cache = _append_both(layer, table, k, v, slots)
    assert np.array_equal(layer.cache.cpu().numpy(), cache)


def test_append_rewrites_one_slot_of_a_pair(table):
    """Value codes of slots 2j, 2j + 1 share a pair row: writing one slot
    again (here with other vectors, some in the same call as their partner)
    replaces its codes and keeps the partner's."""
    spec = _spec("bgpair", ctx=40)
    layer = BgtqLayer(spec, 0, codebooks=table)
    k, v = layer.history_kv(0, device="cpu")
    slots = inputs.slot_mapping(layer.block_table[0].cpu(), history_positions(spec))
    cache = _append_both(layer, table, k, v, slots)
    g = torch.Generator().manual_seed(5)
    pick = torch.tensor([3, 4, 9, 20, 21, 30])
    k2 = (torch.randn(len(pick), *k.shape[1:], generator=g) * 2).to(k.dtype)
    v2 = torch.randn(len(pick), *v.shape[1:], generator=g).to(v.dtype)
    layer.append(k2.cuda(), v2.cuda(), slots[pick].cuda().contiguous())
    torch.cuda.synchronize()
    bgtq.append(cache, _f32(k2), _f32(v2), slots[pick].numpy(), layer.widths_np, layer.v_bits, layer.total_bits,
                _pis(layer), table)
    assert np.array_equal(layer.cache.cpu().numpy(), cache)


def test_library_codebooks_give_the_same_cache(table):
    spec = _spec("bglib", ctx=24)
    a = BgtqLayer(spec, 0)                         # library Lloyd-Max codebooks
    b = BgtqLayer(spec, 0, codebooks=table)        # oracle codebooks
    k, v = a.history_kv(0)
    slots = a.slots(0, history_positions(spec))
    a.append(k, v, slots)
    b.append(k, v, slots)
    torch.cuda.synchronize()
    assert torch.equal(a.cache, b.cache)


@pytest.mark.parametrize("h_q,h_kv,ctxs,splits", [
    (8, 2, [100], 0),
    (4, 1, [1], 0),
    (16, 2, [17, 260, 33], 3),
    (32, 4, [129, 64], 0),
    (16, 2, [50], 40),
    (8, 2, [0, 37, 16], 0),   # an empty sequence, an odd tail (half a slot pair), a whole page
    (64, 8, [33, 0], 2),      # GQA 8 over 8 KV heads with an empty second sequence
])
def test_decode_vs_oracle(table, h_q, h_kv, ctxs, splits):
    B = len(ctxs)
    spec = _spec(f"bgdec{h_q}{h_kv}{B}", h_q=h_q, h_kv=h_kv, batch=B, ctx=max(ctxs), permute=True)
    layer = BgtqLayer(spec, 0, codebooks=table, extra_pages=2)
    cache = bgtq.new_cache(layer.num_pages, h_kv, layer.total_bits, layer.v_bits)
    bt = layer.block_table.cpu().numpy()
    pis = _pis(layer)
    for b, T in enumerate(ctxs):
        k, v = layer.history_kv(b, device="cpu")
        k, v = k[:T], v[:T]
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        bgtq.append(cache, _f32(k), _f32(v), slots, layer.widths_np, layer.v_bits, layer.total_bits, pis, table)
    layer.cache.copy_(torch.as_tensor(cache))
    q = layer.queries()
    cl = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    out = torch.full((B, h_q, 128), float("nan"), device="cuda")
    ws = layer.workspace(splits)
    layer.decode(q, out, ws, splits, context_lens=cl)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    ref = bgtq.decode(q.cpu().double().numpy(), cache, bt, ctxs, layer.widths_np, layer.v_bits, layer.total_bits,
                      pis, table, layer.scale, h_kv)
    for b in range(B):
        _close(out[b].cpu().numpy(), ref[b])


@pytest.mark.parametrize("avg_bits,v_bits,b_max,h_q", [(2, 2, 8, 8), (1, 1, 8, 8), (8, 8, 8, 16), (4, 5, 6, 16),
                                                     (3, 4, 8, 8), (3, 6, 8, 16), (3, 7, 8, 8)])
def test_decode_value_widths(table, avg_bits, v_bits, b_max, h_q):
    """Every value width has its own kernel instance (groups up to 4 and of 8)."""
    ctxs = [70, 33]
    spec = _spec(f"bgvw{avg_bits}{v_bits}{h_q}", h_q=h_q, h_kv=2, batch=2, ctx=max(ctxs), avg_bits=avg_bits,
                 v_bits=v_bits, b_max=b_max, permute=True)
    layer = BgtqLayer(spec, 0, codebooks=table)
    cache = bgtq.new_cache(layer.num_pages, 2, layer.total_bits, layer.v_bits)
    bt = layer.block_table.cpu().numpy()
    pis = _pis(layer)
    for b, T in enumerate(ctxs):
        k, v = layer.history_kv(b, device="cpu")
        slots = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(T)])
        bgtq.append(cache, _f32(k[:T]), _f32(v[:T]), slots, layer.widths_np, layer.v_bits, layer.total_bits, pis,
                    table)
    layer.cache.copy_(torch.as_tensor(cache))
    q = layer.queries()
    cl = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    out = torch.full((2, h_q, 128), float("nan"), device="cuda")
    ws = layer.workspace()
    layer.decode(q, out, ws, 0, context_lens=cl)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    ref = bgtq.decode(q.cpu().double().numpy(), cache, bt, ctxs, layer.widths_np, layer.v_bits, layer.total_bits,
                      pis, table, layer.scale, 2)
    for b in range(2):
        _close(out[b].cpu().numpy(), ref[b])


def test_end_to_end_append_then_decode(table):
    spec = _spec("bge2e", h_q=8, h_kv=2, ctx=150)
    layer = BgtqLayer(spec, 0, codebooks=table)
    k, v = layer.history_kv(0, device="cpu")
    k_new, v_new = layer.new_kv(device="cpu")
    k_all, v_all = torch.cat([k, k_new]), torch.cat([v, v_new])
    slots = inputs.slot_mapping(layer.block_table[0].cpu(), torch.arange(spec.ctx))
    cache = _append_both(layer, table, k_all, v_all, slots)
    assert np.array_equal(layer.cache.cpu().numpy(), cache)
    q = layer.queries()
    out = torch.zeros(1, 8, 128, device="cuda")
    ws = layer.workspace()
    layer.decode(q, out, ws)
    torch.cuda.synchronize()
    ref = bgtq.decode(q.cpu().double().numpy(), cache, layer.block_table.cpu().numpy(), [spec.ctx],
                      layer.widths_np, layer.v_bits, layer.total_bits, _pis(layer), table, layer.scale, 2)
    _close(out.cpu().numpy()[0], ref[0])


def test_bad_widths_are_reported(table):
    spec = _spec("bgbad", ctx=20)
    layer = BgtqLayer(spec, 0, codebooks=table)
    layer.widths[0, 3] = 9
    k, v = layer.history_kv(0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer.append(k, v, layer.slots(0, history_positions(spec)), err)
    torch.cuda.synchronize()
    assert int(err.item()) >= 1
    out = torch.zeros(1, 8, 128, device="cuda")
    ws = layer.workspace()
    layer.decode(layer.queries(), out, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == -1
    assert torch.isfinite(out).all()


def test_full_size_k3v3_sampled(table):
    """The Block-GTQ K3V3 workload at 128K context: GPU prefill and decode of
    all 8 KV heads; codes of sampled tokens bit-exact; sampled heads'
    attention against the oracle (fp64-rotation path for the 128K tokens)."""
    spec = inputs.SPECS["bgtq"]
    layer = BgtqLayer(spec, 0, codebooks=table)
    layer.prefill()
    k_new, v_new = layer.new_kv()
    layer.append(k_new, v_new, layer.new_slots())
    q = layer.queries()
    out = torch.zeros(1, spec.h_q, 128, device="cuda")
    ws = layer.workspace()
    layer.decode(q, out, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    got = out.cpu().numpy()[0]
    pis = _pis(layer)
    bt = layer.block_table.cpu().numpy()
    rng = np.random.default_rng(4)
    k_hist, v_hist = layer.history_kv(0)
    lay = bgtq.tile_layout(layer.total_bits, layer.v_bits)
    for h in (1, 6):
        k = torch.cat([k_hist[:, h], k_new[:, h]])
        v = torch.cat([v_hist[:, h], v_new[:, h]])
        kf, vf = _f32(k), _f32(v)
        T = spec.ctx
        slots = np.array([bt[0, t // 16] * 16 + t % 16 for t in range(T)])
        idx = np.sort(rng.choice(T, size=48, replace=False))
        small = bgtq.new_cache(layer.num_pages, 1, layer.total_bits, layer.v_bits)
        bgtq.append(small, kf[idx][:, None], vf[idx][:, None], slots[idx], layer.widths_np[h:h + 1], layer.v_bits,
                    layer.total_bits, pis, table)
        gpu = layer.cache[:, h].cpu().numpy()
        for t in idx:
            page, s = divmod(int(slots[t]), 16)
            for off, n in ((lay["kb"] * s, lay["kb"]), (lay["k_norms"] + 16 * s, 16), (lay["v_norms"] + 2 * s, 2)):
                assert np.array_equal(gpu[page, off:off + n], small[page, 0, off:off + n]), (h, t)
            # value codes share a pair row with the partner slot: compare this slot's
            assert np.array_equal(bgtq.read_v_codes(gpu[page], s, layer.total_bits, layer.v_bits),
                                  bgtq.read_v_codes(small[page, 0], s, layer.total_bits, layer.v_bits)), (h, t)
        kh, vh = bgtq.dequantize_dense(kf, vf, layer.widths_np[h], layer.v_bits, pis, table, exact_chain=False)
        g = spec.g
        ref = attention.gqa_decode(q[0, h * g:(h + 1) * g].cpu().double().numpy(), kh[:, None], vh[:, None],
                                   float(np.float32(layer.scale)))
        _close(got[h * g:(h + 1) * g], ref)
