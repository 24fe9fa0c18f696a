"""Exact IEEE helpers for decisions taken in the kernel's precision.

A quantisation code is an integer decided by comparing a floating-point
value with thresholds.  For codes to be bit-exact, the oracle decides them
from the same fp32 value the kernel forms.  The kernels form rotated vectors
with a fixed-order chain of fp32 fused multiply-adds (acc = fma(x_i, M_ij,
acc) for i = 0..n-1); this module reproduces that chain exactly.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""
from __future__ import annotations

import numpy as np

F16_MAX = 65504.0


def _two_sum(a: np.ndarray, b: np.ndarray):
    """Knuth's error-free transformation: a + b == s + e exactly (fp64)."""
    s = a + b
    bb = s - a
    e = (a - (s - bb)) + (b - bb)
    return s, e


def fma_f32(a, b, c) -> np.ndarray:
    """Correctly rounded fp32 fused multiply-add round_f32(a*b + c).

    a, b, c are fp32 arrays (broadcastable).  The product of two fp32 values
    is exact in fp64; the sum with c is split into s + e exactly; s rounds to
    fp32 like s + e except when s sits exactly on a midpoint between two fp32
    values, where the sign of e decides the direction.
    """
    a = np.asarray(a, dtype=np.float32).astype(np.float64)
    b = np.asarray(b, dtype=np.float32).astype(np.float64)
    c = np.asarray(c, dtype=np.float32).astype(np.float64)
    p = a * b
    s, e = _two_sum(p, c)
    r = s.astype(np.float32)
    rd = r.astype(np.float64)
    up = np.nextafter(r, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(r, np.float32(-np.inf)).astype(np.float64)
    mid_up = (rd + up) * 0.5          # exact in fp64
    mid_dn = (rd + dn) * 0.5
    go_up = (s == mid_up) & (e > 0)
    go_dn = (s == mid_dn) & (e < 0)
    r = np.where(go_up, np.nextafter(r, np.float32(np.inf)), r)
    r = np.where(go_dn, np.nextafter(r, np.float32(-np.inf)), r)
    return r.astype(np.float32)


def chain_matvec_f32(x: np.ndarray, m: np.ndarray) -> np.ndarray:
    """Row vector(s) times matrix in fp32 as the kernels form it:
    y_j = fma(x_{n-1}, m_{n-1,j}, ... fma(x_1, m_1j, fma(x_0, m_0j, 0)) ...).

    x: [..., n] fp32, m: [n, k] fp32 -> [..., k] fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    m = np.asarray(m, dtype=np.float32)
    acc = np.zeros(x.shape[:-1] + (m.shape[1],), dtype=np.float32)
    for i in range(m.shape[0]):
        acc = fma_f32(x[..., i:i + 1], m[i][None, :] if x.ndim > 1 else m[i], acc)
    return acc


def chain_sumsq_f32(x: np.ndarray) -> np.ndarray:
    """sum_i x_i^2 as the fp32 fma chain in coordinate order. x: [..., n]."""
    x = np.asarray(x, dtype=np.float32)
    acc = np.zeros(x.shape[:-1], dtype=np.float32)
    for i in range(x.shape[-1]):
        acc = fma_f32(x[..., i], x[..., i], acc)
    return acc


def f16_rn_sat(x) -> np.ndarray:
    """fp32 -> fp16 with round-to-nearest-even, saturating to +-65504
    (overflow gives the largest finite value instead of infinity)."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    h = np.where(np.isinf(h) & ~np.isinf(x), np.sign(x) * np.float16(F16_MAX), h)
    return h.astype(np.float16)
