"""Output-space error of the rotated INT2 cache, measured on the GPU.

"Output-Aware Rotation for INT2 KV-Cache Quantization" §3.2 separates the
reconstruction error of the cache, Eq. (9),
    E_rec = ||K - K~||_F^2 + ||V - V~||_F^2,
from the error the model sees after attention and W_O, Eq. (10),
    E_out = sum_j ||y~_j - y_j||^2,   y_j = (sum_s p_s v_s) W_{O,j}^T,
which Eq. (8) splits into a key-induced term (the attention map moves) and
a value-induced term.  This module measures both for a choice of rotation
R (identity, the normalised Hadamard matrix, or the Hadamard matrix times a
seeded Haar orthogonal, the form the library's workloads use) and of the
clip ratio c, with a seeded random W_O.  Learning R from E_out, as the
paper does, is not part of this build.

The cache is written by kvq_append_int2_clip and read back by
kvq_dequant_int2; the quantised output y~ comes from the fused decode
(kvq_decode_attn_int2).  Only the exact reference attention, the change of
basis back (K~ = Z~ R^T + mu, V~ = W~ R^T), the W_O projection and the
norms are plain torch fp64 reductions.

    python -m bit_kv_cache_13_gb300.diagnostics   # prints the table
"""
from __future__ import annotations

import json
import math

import numpy as np
import torch

from . import _lib, inputs
from .workload import Int2Layer, history_positions

ROTATIONS = ("identity", "hadamard", "hadamard_haar")


def head_rotations(kind: str, spec, layer: int, side: str) -> np.ndarray:
    """[H_kv, d, d] fp64 rotations of one kind for one side ("Rk" / "Rv")."""
    d = spec.d
    if kind == "identity":
        return np.stack([np.eye(d)] * spec.h_kv)
    if kind == "hadamard":
        return np.stack([inputs.sylvester_hadamard(d) / math.sqrt(d)] * spec.h_kv)
    if kind == "hadamard_haar":
        return np.stack([inputs.head_rotation(d, spec.name, layer, h, side) for h in range(spec.h_kv)])
    raise ValueError(kind)


def w_out(spec, d_model: int, layer: int = 0, device="cuda") -> torch.Tensor:
    """Seeded random W_O: [H_q, d_model, d] fp64, entries N(0, 1/(H_q d))."""
    g = inputs.torch_gen("cpu", spec.name, layer, "W_O")
    w = torch.randn((spec.h_q, d_model, spec.d), generator=g, dtype=torch.float64)
    return (w / math.sqrt(spec.h_q * spec.d)).to(device)


def output_error(spec, rotation: str, clip: float = 1.0, d_model: int = 4096, layer: int = 0,
                 device="cuda") -> dict:
    """E_rec, E_out and the key / value parts of E_out for sequence 0 of one
    layer of `spec` (all its KV heads), with the given rotation and clip."""
    L = Int2Layer(spec, layer, device=device)
    rk64 = head_rotations(rotation, spec, layer, "Rk")
    rv64 = head_rotations(rotation, spec, layer, "Rv")
    L.R_k = torch.as_tensor(rk64, dtype=torch.float32, device=device).contiguous()
    L.R_v = torch.as_tensor(rv64, dtype=torch.float32, device=device).contiguous()
    k, v = L.history_kv(0)                                   # [T, H_kv, d] bf16
    T = k.shape[0]
    L.mu = inputs.key_centre(k).to(device).contiguous()
    slots = L.slots(0, history_positions(spec)).contiguous()
    _lib.kvq_append_int2_clip(k.contiguous(), v.contiguous(), slots, L.mu, L.R_k, L.R_v, clip, L.cache,
                              L.num_pages)
    zk = torch.empty((T, spec.h_kv, spec.d), dtype=torch.float32, device=device)
    zv = torch.empty_like(zk)
    _lib.kvq_dequant_int2(L.cache, L.num_pages, spec.h_kv, slots, zk, zv)

    f64 = torch.float64
    rk = L.R_k.to(f64)
    rv = L.R_v.to(f64)
    K, V = k.to(f64), v.to(f64)
    Kt = torch.einsum("thi,hji->thj", zk.to(f64), rk) + L.mu.to(f64)     # Z~ R_k^T + mu
    Vt = torch.einsum("thi,hji->thj", zv.to(f64), rv)                    # W~ R_v^T
    e_rec = float(((K - Kt) ** 2).sum() + ((V - Vt) ** 2).sum())

    # queries of sequence 0 and the fused decode over the T cached tokens
    q = L.queries()[:1].contiguous()                          # [1, H_q, d] bf16
    out = torch.zeros((1, spec.h_q, spec.d), dtype=torch.float32, device=device)
    ws = L.workspace()
    ctx = torch.tensor([T], dtype=torch.int32, device=device)
    _lib.kvq_decode_attn_int2(q, L.cache, L.num_pages, L.block_table[:1].contiguous(), ctx, L.R_k, L.R_v,
                              L.scale, out, ws)
    torch.cuda.synchronize()
    if _lib.kvq_workspace_status(ws) != 0:
        raise RuntimeError("decode reported an error")

    w_o = w_out(spec, d_model, layer, device)
    g = spec.h_q // spec.h_kv
    sc = float(np.float32(L.scale))
    e_out = e_key = e_val = 0.0
    qd = q[0].to(f64)
    for j in range(spec.h_q):
        h = j // g
        p = torch.softmax(K[:, h] @ qd[j] * sc, dim=0)          # Eqs. (1)-(2)
        pt = torch.softmax(Kt[:, h] @ qd[j] * sc, dim=0)        # Eq. (5)
        y = (p @ V[:, h]) @ w_o[j].T
        y_fused = out[0, j].to(f64) @ w_o[j].T                  # Eq. (7), from the kernel
        e_out += float(((y_fused - y) ** 2).sum())
        e_key += float(((((pt - p) @ V[:, h]) @ w_o[j].T) ** 2).sum())      # Eq. (8)
        e_val += float((((pt @ (Vt[:, h] - V[:, h])) @ w_o[j].T) ** 2).sum())
    return {"rotation": rotation, "clip": clip, "tokens": T, "kv_heads": spec.h_kv, "d_model": d_model,
            "E_rec": e_rec, "E_out": e_out, "E_out_key": e_key, "E_out_value": e_val}


def table(spec_name: str = "llama8b_diag", clips=(1.0, 0.95, 0.9, 0.85), device="cuda"):
    """Rows of output_error over the three rotations and the clip ratios for
    a one-layer, 4096-token Llama-3-8B-shaped workload (32 q / 8 KV heads,
    keys with heavy-offset channels and RoPE, values with outlier channels)."""
    spec = inputs.small_spec(spec_name, h_q=32, h_kv=8, batch=1, ctx=4097, k_kind="offset_rope",
                             v_kind="outlier10pct2", permute=True)
    return [output_error(spec, rot, c, device=device) for rot in ROTATIONS for c in clips]


if __name__ == "__main__":
    for row in table():
        print(json.dumps({k: (round(v, 6) if isinstance(v, float) else v) for k, v in row.items()}))
