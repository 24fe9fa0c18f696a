"""Seeded synthetic workloads for the rotated low-bit KV-cache path.

This module only draws inputs: query/key/value activations, per-head
rotations, key centres, RoPE-block energy scores, TQ rotations and paged
block tables.  It holds none of the quantisation or attention arithmetic;
both the CUDA library and the fp64 reference checker consume what it
produces.

Distributions follow the five workloads of the method's evaluation set-up
(rotation-based INT2 KV-cache quantisation, "Output-Aware Rotation for INT2
KV-Cache Quantization" §3; RoPE-aware bit allocation, "RoPE-Aware Bit
Allocation for KV-Cache Quantization", method steps (1)-(4)):

  tiny     1 layer, 1 KV head, 4 q heads, B=1, 256 cached + 1 decode token
  llama8b  32 q / 8 KV heads, B=8, 32K context, post-RoPE keys (theta 5e5)
  qwen8b   36 layers x (32 q / 8 KV), B=1, 128K context
  bgtq     32 q / 8 KV, B=1, 128K, block energies lognormal(0, 2)
  sweep70b 64 q / 8 KV (GQA 8), B in {1,8,32,64} x T in {4K,32K,128K}

Small workloads are drawn on the CPU; large ones on the device with a
seeded torch generator (sampled slices are copied back for checking).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 20261202
HEAD_DIM = 128
PAGE_SIZE = 16


def derive_seed(*keys) -> int:
    """Stable 63-bit seed from SEED_BASE and any tuple of keys."""
    h = hashlib.sha256(repr((SEED_BASE,) + tuple(keys)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def np_rng(*keys) -> np.random.Generator:
    return np.random.default_rng(derive_seed(*keys))


def torch_gen(device, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(derive_seed(*keys))
    return g


# --------------------------------------------------------------------------
# rotations (parameters of the method; here seeded instead of learned)
# --------------------------------------------------------------------------

def sylvester_hadamard(n: int) -> np.ndarray:
    """+-1 Hadamard matrix of order n (a power of two), Sylvester construction."""
    assert n >= 1 and n & (n - 1) == 0
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def haar_orthogonal(n: int, *keys) -> np.ndarray:
    """Haar-distributed orthogonal matrix: QR of a Gaussian matrix with the
    column signs fixed by the signs of diag(R)."""
    a = np_rng("haar", n, *keys).standard_normal((n, n))
    q, r = np.linalg.qr(a)
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def head_rotation(d: int, *keys) -> np.ndarray:
    """Per-head orthogonal R = (H_d / sqrt(d)) @ Q, with Q a seeded Haar
    orthogonal standing in for the learned per-head correction.  fp64."""
    return (sylvester_hadamard(d) / np.sqrt(d)) @ haar_orthogonal(d, "corr", *keys)


def tq_rotations(max_n: int = HEAD_DIM, *keys):
    """One shared Haar orthogonal Pi_n per even sub-vector length n <= max_n.

    Returns (table_f64, offsets) where Pi_n occupies
    table[offsets[n] : offsets[n] + n*n] row-major; offsets[n] = -1 for odd n.
    """
    offsets = np.full(max_n + 1, -1, dtype=np.int64)
    chunks, pos = [], 0
    for n in range(2, max_n + 1, 2):
        offsets[n] = pos
        m = haar_orthogonal(n, "tq", *keys)
        chunks.append(m.reshape(-1))
        pos += n * n
    return np.concatenate(chunks), offsets


# --------------------------------------------------------------------------
# bf16 helpers
# --------------------------------------------------------------------------

def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round to bfloat16 (round-to-nearest-even)."""
    return x.to(torch.bfloat16)


def bf16_to_f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").to(torch.float64).numpy()


# --------------------------------------------------------------------------
# workload specs
# --------------------------------------------------------------------------

@dataclass
class Spec:
    name: str
    n_layers: int
    h_q: int
    h_kv: int
    batch: int
    ctx: int                     # tokens attended after the decode-step append
    k_kind: str                  # "outlier_offset" | "offset_rope" | "energy_rope"
    v_kind: str                  # "outlier20" | "outlier10pct2"
    d: int = HEAD_DIM
    rope_theta: float = 500000.0
    permute_pages: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def g(self) -> int:
        return self.h_q // self.h_kv

    @property
    def pages_per_seq(self) -> int:
        return (self.ctx + PAGE_SIZE - 1) // PAGE_SIZE


SPECS = {
    "tiny": Spec("tiny", 1, 4, 1, 1, 257, "outlier_offset", "outlier20"),
    "llama8b": Spec("llama8b", 1, 32, 8, 8, 32768, "offset_rope", "outlier20",
                    permute_pages=True),
    "qwen8b": Spec("qwen8b", 36, 32, 8, 1, 131072, "outlier_offset", "outlier10pct2",
                   permute_pages=True),
    "bgtq": Spec("bgtq", 1, 32, 8, 1, 131072, "energy_rope", "gauss",
                 permute_pages=True, extra={"avg_bits": 3, "v_bits": 3,
                                            "b_min": 1, "b_max": 8}),
}


# BF16 window of the window workload: sink and recent tokens per sequence
WINDOW_SINK, WINDOW_RECENT = 4, 128


def sweep70b_spec(batch: int, ctx: int) -> Spec:
    return Spec(f"sweep70b_b{batch}_t{ctx}", 1, 64, 8, batch, ctx,
                "outlier_offset", "outlier20", permute_pages=True)


def small_spec(name, *, h_q=4, h_kv=1, batch=1, ctx=257, n_layers=1,
               k_kind="outlier_offset", v_kind="outlier20", permute=False, **extra):
    """A reduced workload with the distributions of the named ones (used by
    the parity tests to cover ragged tails, several tiles and GQA shapes)."""
    return Spec(name, n_layers, h_q, h_kv, batch, ctx, k_kind, v_kind,
                permute_pages=permute, extra=dict(extra))


# --------------------------------------------------------------------------
# per-(layer, head) distribution parameters (small, numpy-seeded)
# --------------------------------------------------------------------------

def _outlier_channels(spec, layer, head, tensor, count):
    return np.sort(np_rng(spec.name, layer, head, tensor, "outliers")
                   .choice(spec.d, size=count, replace=False))


def key_params(spec: Spec, layer: int, head: int):
    """Returns (scale[d], offset[d]) applied as k = z*scale + offset with
    z ~ N(0,1) (pre-RoPE for the RoPE workloads)."""
    d = spec.d
    scale = np.ones(d)
    offset = np.zeros(d)
    if spec.k_kind == "outlier_offset":
        scale[_outlier_channels(spec, layer, head, "k", 4)] = 20.0
        offset = np_rng(spec.name, layer, head, "k", "offset").normal(0.0, 2.0, d)
    elif spec.k_kind == "offset_rope":
        rng = np_rng(spec.name, layer, head, "k", "heavy")
        ch = np.sort(rng.choice(d, size=8, replace=False))
        offset[ch] = 10.0 * rng.choice([-1.0, 1.0], size=8)
    elif spec.k_kind == "energy_rope":
        s = block_energies(spec, layer, head)
        L = d // 2
        sd = np.sqrt(s / 2.0)
        scale[:L] = sd
        scale[L:] = sd
    else:
        raise ValueError(spec.k_kind)
    return scale, offset


def value_params(spec: Spec, layer: int, head: int):
    d = spec.d
    scale = np.ones(d)
    if spec.v_kind == "outlier20":
        scale[_outlier_channels(spec, layer, head, "v", 4)] = 20.0
    elif spec.v_kind == "outlier10pct2":
        n = int(round(0.02 * d))
        scale[_outlier_channels(spec, layer, head, "v", n)] = 10.0
    elif spec.v_kind == "gauss":
        pass
    else:
        raise ValueError(spec.v_kind)
    return scale


def block_energies(spec: Spec, layer: int, head: int) -> np.ndarray:
    """Per-RoPE-block energy scores s_i ~ lognormal(0, sigma=2), i < d/2."""
    return np_rng(spec.name, layer, head, "energy").lognormal(0.0, 2.0, spec.d // 2)


def query_params(spec: Spec, layer: int, head_kv: int):
    if spec.k_kind == "energy_rope":
        s = block_energies(spec, layer, head_kv)
        sd = np.sqrt(s / 2.0)
        return np.concatenate([sd, sd])
    return np.ones(spec.d)


# --------------------------------------------------------------------------
# RoPE (input preparation: the kernels consume post-RoPE keys)
# --------------------------------------------------------------------------

def rope_apply(x: torch.Tensor, positions: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half RoPE: block i pairs dims (i, i + d/2) and turns by
    pos * theta^(-2i/d).  x: [..., n, d] float, positions: [n]."""
    d = x.shape[-1]
    L = d // 2
    inv = theta ** (-2.0 * torch.arange(L, dtype=torch.float64, device=x.device) / d)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    shape = [1] * (x.dim() - 2) + [positions.numel(), L]
    c, s = c.reshape(shape), s.reshape(shape)
    xd = x.to(torch.float64)
    a, b = xd[..., :L], xd[..., L:]
    return torch.cat([a * c - b * s, a * s + b * c], dim=-1).to(x.dtype)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------

def _scaled(z: torch.Tensor, scale: np.ndarray, offset=None) -> torch.Tensor:
    sc = torch.as_tensor(scale, dtype=z.dtype, device=z.device)
    out = z * sc
    if offset is not None:
        out = out + torch.as_tensor(offset, dtype=z.dtype, device=z.device)
    return out


def gen_keys(spec: Spec, layer: int, batch_idx: int, positions: torch.Tensor,
             device="cpu", tag="hist") -> torch.Tensor:
    """Keys [n, H_kv, d] bf16 for one sequence at the given positions."""
    n = positions.numel()
    out = torch.empty((n, spec.h_kv, spec.d), dtype=torch.bfloat16, device=device)
    for h in range(spec.h_kv):
        g = torch_gen(device, spec.name, layer, batch_idx, h, "k", tag)
        z = torch.randn((n, spec.d), generator=g, device=device, dtype=torch.float32)
        scale, offset = key_params(spec, layer, h)
        k = _scaled(z, scale, offset)
        if spec.k_kind in ("offset_rope", "energy_rope"):
            k = rope_apply(k, positions.to(device), spec.rope_theta)
        out[:, h] = to_bf16(k)
    return out


def gen_values(spec: Spec, layer: int, batch_idx: int, n: int, device="cpu",
               tag="hist") -> torch.Tensor:
    out = torch.empty((n, spec.h_kv, spec.d), dtype=torch.bfloat16, device=device)
    for h in range(spec.h_kv):
        g = torch_gen(device, spec.name, layer, batch_idx, h, "v", tag)
        z = torch.randn((n, spec.d), generator=g, device=device, dtype=torch.float32)
        out[:, h] = to_bf16(_scaled(z, value_params(spec, layer, h)))
    return out


def gen_prefix_queries(spec: Spec, layer: int, positions: torch.Tensor, device="cpu") -> torch.Tensor:
    """Queries [n, H_q, d] bf16 of a calibration prefix at the given
    positions (post-RoPE for the RoPE workloads), drawn like the decode
    queries: per-block standard deviations from the head's energy scores."""
    n = positions.numel()
    out = torch.empty((n, spec.h_q, spec.d), dtype=torch.bfloat16, device=device)
    for j in range(spec.h_q):
        g = torch_gen(device, spec.name, layer, j, "qcal")
        z = torch.randn((n, spec.d), generator=g, device=device, dtype=torch.float32)
        z = _scaled(z, query_params(spec, layer, j // spec.g))
        if spec.k_kind in ("offset_rope", "energy_rope"):
            z = rope_apply(z, positions.to(device), spec.rope_theta)
        out[:, j] = to_bf16(z)
    return out


def gen_queries(spec: Spec, layer: int, device="cpu") -> torch.Tensor:
    """Decode queries [B, H_q, d] bf16 (post-RoPE at position ctx-1 for the
    RoPE workloads)."""
    q = torch.empty((spec.batch, spec.h_q, spec.d), dtype=torch.bfloat16, device=device)
    pos = torch.tensor([spec.ctx - 1], device=device)
    for b in range(spec.batch):
        for j in range(spec.h_q):
            g = torch_gen(device, spec.name, layer, b, j, "q")
            z = torch.randn((1, spec.d), generator=g, device=device, dtype=torch.float32)
            z = _scaled(z, query_params(spec, layer, j // spec.g))
            if spec.k_kind in ("offset_rope", "energy_rope"):
                z = rope_apply(z, pos, spec.rope_theta)
            q[b, j] = to_bf16(z[0])
    return q


def key_centre(keys_bf16: torch.Tensor, n_calib: int = 512) -> torch.Tensor:
    """Offline per-head key centre mu_h: channel mean of the first
    min(T, n_calib) keys, accumulated in fp64, returned fp32 [H_kv, d]."""
    k = keys_bf16[: min(keys_bf16.shape[0], n_calib)].to(torch.float64)
    return k.mean(dim=0).to(torch.float32)


# --------------------------------------------------------------------------
# paging
# --------------------------------------------------------------------------

def block_tables(spec: Spec, n_pages_total: int | None = None, device="cpu"):
    """Physical page ids [B, pages_per_seq] int32.  Pages of all sequences are
    drawn from one pool, randomly permuted when the workload asks for it."""
    pps = spec.pages_per_seq
    total = spec.batch * pps if n_pages_total is None else n_pages_total
    assert total >= spec.batch * pps
    if spec.permute_pages:
        perm = np_rng(spec.name, "pages").permutation(total)[: spec.batch * pps]
    else:
        perm = np.arange(spec.batch * pps)
    return torch.as_tensor(perm.reshape(spec.batch, pps).astype(np.int32), device=device)


def slot_mapping(block_table_row: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    """slot = page * 16 + offset for each token position of one sequence."""
    pages = block_table_row.to(torch.int64)[positions // PAGE_SIZE]
    return (pages * PAGE_SIZE + positions % PAGE_SIZE).to(torch.int32)
