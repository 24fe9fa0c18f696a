"""GQA decode attention in fp64 (TEST INFRASTRUCTURE ONLY).

Output-Aware Rotation for INT2 KV-Cache Quantization, §3 "Preliminaries",
Eqs. (1)-(2): for query head j in G_h (the query heads sharing KV head h),
    a_{t,s} = <q_{t,j}, k_{s,h}> / sqrt(d),   p_t = softmax_{s<=t}(a_{t,s}),
    o_{t,j} = sum_{s<=t} p_{t,s} v_{s,h}.
Query heads are grouped contiguously: j belongs to KV head j // (H_q / H_kv).
"""
from __future__ import annotations

import numpy as np


def softmax(a: np.ndarray) -> np.ndarray:
    """Softmax over the last axis in fp64 (max-shifted)."""
    a = np.asarray(a, dtype=np.float64)
    m = a.max(axis=-1, keepdims=True)
    e = np.exp(a - m)
    return e / e.sum(axis=-1, keepdims=True)


def gqa_decode(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """One decode query per head against a cache.

    q: [H_q, d]; keys, values: [T, H_kv, d]; returns o: [H_q, d] (fp64).
    T == 0 gives zeros (nothing to attend).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    h_q, d = q.shape
    T, h_kv, _ = keys.shape
    out = np.zeros((h_q, d))
    if T == 0:
        return out
    g = h_q // h_kv
    for j in range(h_q):
        h = j // g
        a = keys[:, h, :] @ q[j] * scale          # Eq. (1)
        p = softmax(a)
        out[j] = p @ values[:, h, :]             # Eq. (2)
    return out
