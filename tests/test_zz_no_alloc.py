"""The allocation-free INT2 decode entry point gives the same output as the
workspace entry point.

kvq_decode_attn_int2_noalloc exists for callers that cannot allocate device
memory when they call the library (a serving loop with all device memory
planned up front, or a host that owns every device allocation), so it keeps
its split-K scratch in a fixed array inside the library.  This file runs
last so that a failure here never hides the other tests.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _layer(name, h_q, h_kv, batch, ctx):
    spec = inputs.small_spec(name, h_q=h_q, h_kv=h_kv, batch=batch, ctx=ctx, permute=True)
    layer = Int2Layer(spec, 0)
    layer.prefill()
    return layer


def _both(layer, q, splits):
    spec = layer.spec
    ref = torch.zeros((spec.batch, spec.h_q, 128), dtype=torch.float32, device="cuda")
    ws = layer.workspace(splits)
    _lib.kvq_decode_attn_int2(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens, layer.R_k,
                              layer.R_v, layer.scale, ref, ws, splits)
    got = torch.full_like(ref, float("nan"))
    _lib.kvq_decode_attn_int2_noalloc(q, layer.cache, layer.num_pages, layer.block_table, layer.context_lens,
                                      layer.R_k, layer.R_v, layer.scale, got, splits)
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    a = _layer("noalloc_a", 32, 8, 2, 3000)
    b = _layer("noalloc_b", 8, 2, 3, 777)
    calls = [(a, 0), (b, 5), (a, 0)]              # two shapes back to back, then the first again
    for layer, splits in calls:
        q = layer.queries()
        got, ref = _both(layer, q, splits)
        assert np.all(np.isfinite(got))
        err = np.max(np.abs(got - ref))
        assert err <= TOL * np.max(np.abs(ref)), err


def test_noalloc_gqa8_and_the_largest_shape_that_fits():
    """The 8-warp GQA-8 instance through the fixed scratch, and the largest
    batch of 64 q / 8 KV heads at 4K context whose partials fit 4 MiB (one
    more sequence is refused)."""
    a = _layer("noalloc_g8", 64, 8, 2, 2500)
    got, ref = _both(a, a.queries(), 0)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= TOL * np.max(np.abs(ref))
    big = _layer("noalloc_big", 64, 8, 62, 4096)
    got, ref = _both(big, big.queries(), 0)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= TOL * np.max(np.abs(ref))
    q = torch.zeros((63, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((63, 64, 128), dtype=torch.float32, device="cuda")
    bt = torch.zeros((63, 256), dtype=torch.int32, device="cuda")
    cl = torch.full((63,), 4096, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.KvqError) as e:
        _lib.kvq_decode_attn_int2_noalloc(q, big.cache, big.num_pages, bt, cl, big.R_k, big.R_v, 0.1, out)
    assert e.value.status == -3 and "scratch" in str(e.value)


def test_noalloc_rejects_shapes_above_its_scratch():
    q = torch.zeros((64, 64, 128), dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    bt = torch.zeros((64, 8192), dtype=torch.int32, device="cuda")
    cl = torch.zeros(64, dtype=torch.int32, device="cuda")
    R = torch.zeros((8, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.zeros((64, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.KvqError) as e:
        _lib.kvq_decode_attn_int2_noalloc(q, dummy, 1, bt, cl, R, R, 0.1, out, num_splits=128)
    assert e.value.status == -3
    assert "scratch" in str(e.value)
