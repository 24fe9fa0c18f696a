"""Failure detection and the dependency contract of the INT2 path, on the
GPU, without faulting it.

* A bounded in-kernel wait that runs out: the test hook makes the next
  decode leave one bulk copy unissued, so its mbarrier phase never
  completes; the kernel gives up after its (shortened) limit, lets its other
  copies land, returns, and the workspace reports KVQ_ERR_CUDA.  The next
  call on the same workspace is correct again.
* Every input may be written by the kernel just before the call: rotations
  copied into place right before an append or a decode are the ones used.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer, history_positions
from oracle import int2

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _layer(name, h_q=4, h_kv=1, batch=1, ctx=300):
    spec = inputs.small_spec(name, h_q=h_q, h_kv=h_kv, batch=batch, ctx=ctx, permute=True)
    layer = Int2Layer(spec, 0)
    layer.prefill()
    return layer


def _decode(layer, q, ws, splits=0):
    out = torch.full((layer.spec.batch, layer.spec.h_q, 128), float("nan"), device="cuda")
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens, layer.R_k,
                              layer.R_v, layer.scale, out, ws, splits)
    return out


@pytest.mark.parametrize("h_q", [8, 16])  # GQA 4 (9-slot rings) and GQA 8 (6-slot rings)
def test_wait_that_runs_out_is_reported_and_the_context_stays_usable(h_q):
    layer = _layer(f"tmo{h_q}", h_q=h_q, h_kv=2, batch=2, ctx=700)
    q = layer.queries()
    ws = layer.workspace()
    good = _decode(layer, q, ws)
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    _lib.kvq_debug_drop_next_copy()
    bad = _decode(layer, q, ws)
    torch.cuda.synchronize()                       # returns: the kernel gave up on its own
    assert _lib.kvq_workspace_status(ws) == -4     # KVQ_ERR_CUDA: an in-kernel wait timed out
    assert "timed out" in _lib.load().kvq_last_error().decode()
    assert int(ws[256:256 + 4 * 4].view(torch.int32).abs().sum()) == 0   # tickets reset all the same
    assert torch.isfinite(bad).all()
    assert not torch.equal(bad, good)              # a page really was left out
    again = _decode(layer, q, ws)                  # the hook is one-shot
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    assert torch.equal(again, good)


@pytest.mark.parametrize("splits", [0, 1])  # with one CTA per unit, CTA 0 (whose copy is dropped) holds the window
def test_window_decode_wait_that_runs_out_still_completes_the_tickets(splits):
    # The CTA whose share ends a unit also attends the unit's BF16 window;
    # after one of its waits runs out it still publishes the window partial,
    # so every unit's ticket completes, is reset, and the next call is exact.
    layer = _layer(f"tmow{splits}", h_q=8, h_kv=2, batch=2, ctx=700)
    q = layer.queries()
    mu = torch.zeros(2, 128, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    kw = torch.randn((2, 16, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    vw = torch.randn((2, 16, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    lens = torch.tensor([16, 9], dtype=torch.int32, device="cuda")
    nbytes = _lib.kvq_decode_workspace_bytes(2, 8, 2, layer.block_table.shape[1], splits + 1 if splits else 0)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

    def win():
        out = torch.full((2, 8, 128), float("nan"), device="cuda")
        _lib.kvq_decode_attn_int2_window(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                         layer.R_k, layer.R_v, mu, kw, vw, lens, layer.scale, out, ws, splits)
        return out

    good = win()
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    _lib.kvq_debug_drop_next_copy()
    bad = win()
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == -4
    assert int(ws[256:256 + 4 * 4].view(torch.int32).abs().sum()) == 0   # tickets reset all the same
    assert torch.isfinite(bad).all()
    assert not torch.equal(bad, good)
    again = win()
    torch.cuda.synchronize()
    assert _lib.kvq_workspace_status(ws) == 0
    assert torch.equal(again, good)


def test_rotations_written_just_before_append_and_decode():
    spec = inputs.small_spec("rwb", h_q=8, h_kv=2, batch=1, ctx=400, permute=True)
    ref = Int2Layer(spec, 0)
    ref.prefill()
    got = Int2Layer(spec, 0)
    R_k, R_v = got.R_k.clone(), got.R_v.clone()
    k, v = got.history_kv(0)
    got.mu = inputs.key_centre(k).cuda().contiguous()
    slots = got.slots(0, history_positions(spec))
    # the rotation buffers hold other values until a kernel on the same
    # stream, issued right before each call, writes the right ones
    got.R_k.zero_()
    got.R_v.fill_(3.0)
    got.R_k.copy_(R_k)
    got.R_v.copy_(R_v)
    _lib.kvq_append_int2(k, v, slots, got.mu, got.R_k, got.R_v, got.cache, got.num_pages)
    torch.cuda.synchronize()
    assert torch.equal(got.cache, ref.cache)
    q = ref.queries()
    want = _decode(ref, q, ref.workspace())
    got.R_k.fill_(-1.0)
    got.R_v.zero_()
    got.R_k.copy_(R_k)
    got.R_v.copy_(R_v)
    out = _decode(got, q, got.workspace())
    torch.cuda.synchronize()
    assert torch.equal(out, want)
