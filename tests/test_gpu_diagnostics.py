"""GPU measurement of the output-space error (E_rec, E_out and its key /
value parts; "Output-Aware Rotation for INT2 KV-Cache Quantization" §3.2,
Eqs. (5)-(10)) against the fp64 oracle, and the INT2 clip ratio and cache
read-back calls it uses.

Bars: clipped caches bit-exact; read-back values bit-exact (one fp32 fma);
E_rec and the Eq. (8) parts <= 1e-9 relative (same codes, fp64 change of
basis in another order); E_out, which takes the fused decode's output,
within 5 % (the kernel's arithmetic error is far below the INT2 error).
"""
import math

import numpy as np
import pytest
import torch

from bit_kv_cache_13_gb300 import _lib, diagnostics, inputs
from bit_kv_cache_13_gb300.workload import Int2Layer, history_positions
from oracle import diagnostics as odiag
from oracle import int2

pytestmark = pytest.mark.gpu


def _spec(name, T=1024):
    return inputs.small_spec(name, h_q=8, h_kv=2, batch=1, ctx=T + 1, k_kind="offset_rope", v_kind="outlier10pct2",
                             permute=True)


@pytest.mark.parametrize("clip", [1.0, 0.9, 0.6])
def test_clipped_append_and_read_back_bit_exact(clip):
    spec = _spec(f"clip{int(clip * 100)}", T=300)
    L = Int2Layer(spec, 0)
    k, v = L.history_kv(0)
    L.mu = inputs.key_centre(k).cuda().contiguous()
    slots = L.slots(0, history_positions(spec)).contiguous()
    _lib.kvq_append_int2_clip(k.contiguous(), v.contiguous(), slots, L.mu, L.R_k, L.R_v, clip, L.cache, L.num_pages)
    zk = torch.empty((k.shape[0], 2, 128), device="cuda")
    zv = torch.empty_like(zk)
    _lib.kvq_dequant_int2(L.cache, L.num_pages, 2, slots, zk, zv)
    torch.cuda.synchronize()
    cache = int2.new_cache(L.num_pages, 2)
    f32 = lambda t: t.detach().cpu().float().numpy()
    int2.append(cache, f32(k), f32(v), slots.cpu().numpy(), f32(L.mu), f32(L.R_k), f32(L.R_v), clip=clip)
    assert np.array_equal(L.cache.cpu().numpy(), cache)
    bt = L.block_table.cpu().numpy()[0]
    for h in range(2):
        for side, got in ((0, zk), (1, zv)):
            n = k.shape[0]
            tiles = cache[bt[: (n + 15) // 16], h]
            off_c = int2.OFF_K_CODES if side == 0 else int2.OFF_V_CODES
            recs = tiles[:, off_c: off_c + 16 * 32].reshape(-1, 32)[:n]
            meta = tiles[:, np.stack([int2.meta_bytes(side, s) for s in range(16)])].reshape(-1, 16)[:n]
            sc, mn = int2.unpack_meta(meta)
            want = int2.dequantize_f32(int2.unpack_codes(recs), sc, mn)
            assert np.array_equal(got[:, h].cpu().numpy(), want)


def test_clip_one_is_the_plain_append():
    spec = _spec("clip_plain", T=200)
    L = Int2Layer(spec, 0)
    k, v = L.history_kv(0)
    mu = inputs.key_centre(k).cuda().contiguous()
    slots = L.slots(0, history_positions(spec)).contiguous()
    a = torch.zeros_like(L.cache)
    b = torch.zeros_like(L.cache)
    _lib.kvq_append_int2(k.contiguous(), v.contiguous(), slots, mu, L.R_k, L.R_v, a, L.num_pages)
    _lib.kvq_append_int2_clip(k.contiguous(), v.contiguous(), slots, mu, L.R_k, L.R_v, 1.0, b, L.num_pages)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    with pytest.raises(_lib.KvqError):
        _lib.kvq_append_int2_clip(k.contiguous(), v.contiguous(), slots, mu, L.R_k, L.R_v, 1.5, b, L.num_pages)


@pytest.mark.parametrize("rotation,clip", [("identity", 1.0), ("hadamard_haar", 1.0), ("hadamard", 0.9)])
def test_output_error_matches_oracle(rotation, clip):
    spec = _spec(f"diag_{rotation}_{int(clip * 100)}")
    d_model = 256
    got = diagnostics.output_error(spec, rotation, clip, d_model=d_model)
    # the same cache, written and read by the oracle
    L = Int2Layer(spec, 0)
    k, v = L.history_kv(0)            # drawn on the device, as the module draws them
    k, v = k.cpu(), v.cpu()
    f32 = lambda t: t.detach().cpu().float().numpy()
    mu = f32(inputs.key_centre(k))
    rk = diagnostics.head_rotations(rotation, spec, 0, "Rk").astype(np.float32)
    rv = diagnostics.head_rotations(rotation, spec, 0, "Rv").astype(np.float32)
    kt = np.zeros((k.shape[0], 2, 128))
    vt = np.zeros_like(kt)
    for h in range(2):
        zk = int2.rotate_keys(f32(k[:, h]), mu[h], rk[h], exact_chain=True)[0]
        zv = int2.rotate_values(f32(v[:, h]), rv[h], exact_chain=True)[0]
        # the fp32 values the library reads back, then the change of basis in fp64
        kt[:, h] = int2.dequantize_f32(*int2.quantize(zk, clip)).astype(np.float64) @ rk[h].astype(np.float64).T + mu[h]
        vt[:, h] = int2.dequantize_f32(*int2.quantize(zv, clip)).astype(np.float64) @ rv[h].astype(np.float64).T
    q = f32(inputs.gen_queries(spec, 0, device="cuda"))[0].astype(np.float64)
    w_o = diagnostics.w_out(spec, d_model, 0, device="cpu").numpy()
    ref = odiag.output_error(q, f32(k), f32(v), kt, vt, w_o, float(np.float32(1 / math.sqrt(128))))
    for key in ("E_rec", "E_out_key", "E_out_value"):
        assert abs(got[key] - ref[key]) <= 1e-9 * ref[key], (key, got[key], ref[key])
    assert abs(got["E_out"] - ref["E_out"]) <= 0.05 * ref["E_out"], (got["E_out"], ref["E_out"])


def test_rotation_lowers_the_reconstruction_error_of_outlier_values():
    # Values with 2 % outlier channels: a rotation spreads the outliers over
    # all channels of a group, so E_rec drops against R = I.
    spec = _spec("diag_rot", T=1024)
    e = {rot: diagnostics.output_error(spec, rot, 1.0, d_model=256)["E_rec"] for rot in diagnostics.ROTATIONS}
    assert e["hadamard"] < e["identity"] and e["hadamard_haar"] < e["identity"]
