"""Output-space error of a quantised KV cache (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows "Output-Aware Rotation for INT2 KV-Cache Quantization" §3.2:
  Eq. (5)  a~ = <q, k~> / sqrt(d), p~ = softmax(a~) over the cached tokens;
  Eq. (6)  the key error moves the logits, Delta a = <q, Delta k> / sqrt(d);
  Eq. (7)  y~_j = (sum_s p~_s v~_s) W_{O,j}^T, head j's output contribution;
  Eq. (8)  Delta y_j = (sum_s Delta p_s v_s) W_{O,j}^T        key-induced
                     + (sum_s p~_s Delta v_s) W_{O,j}^T       value-induced;
  Eq. (9)  E_rec = ||K - K~||_F^2 + ||V - V~||_F^2;
  Eq. (10) E_out = ||y~ - y||^2, here summed over the query heads.
The paper learns a rotation from E_out; that training is out of scope, the
errors themselves are computed here for given effective keys and values.
"""
from __future__ import annotations

import numpy as np

from . import attention


def output_error(q, k, v, k_eff, v_eff, w_o, scale):
    """q [H_q, d]; k, v, k_eff, v_eff [T, H_kv, d] (exact and effective
    cached keys / values, original basis); w_o [H_q, d_model, d] (W_{O,j});
    scale = 1/sqrt(d).  Returns a dict of fp64 scalars
        E_rec, E_out, E_out_key, E_out_value  (||delta y_K||^2, ||delta y_V||^2)
    and the per-head arrays dy, dy_key, dy_value [H_q, d_model]."""
    q = np.asarray(q, np.float64)
    k, v = np.asarray(k, np.float64), np.asarray(v, np.float64)
    kt, vt = np.asarray(k_eff, np.float64), np.asarray(v_eff, np.float64)
    w_o = np.asarray(w_o, np.float64)
    h_q, d = q.shape
    T, h_kv, _ = k.shape
    g = h_q // h_kv
    e_rec = float(np.sum((k - kt) ** 2) + np.sum((v - vt) ** 2))
    dy = np.zeros((h_q, w_o.shape[1]))
    dy_k = np.zeros_like(dy)
    dy_v = np.zeros_like(dy)
    for j in range(h_q):
        h = j // g
        p = attention.softmax(k[:, h] @ q[j] * scale)        # Eqs. (1)-(2)
        pt = attention.softmax(kt[:, h] @ q[j] * scale)      # Eq. (5)
        y = (p @ v[:, h]) @ w_o[j].T
        yt = (pt @ vt[:, h]) @ w_o[j].T                       # Eq. (7)
        dy[j] = yt - y
        dy_k[j] = ((pt - p) @ v[:, h]) @ w_o[j].T             # Eq. (8), key-induced
        dy_v[j] = (pt @ (vt[:, h] - v[:, h])) @ w_o[j].T      # Eq. (8), value-induced
    return {"E_rec": e_rec, "E_out": float(np.sum(dy ** 2)), "E_out_key": float(np.sum(dy_k ** 2)),
            "E_out_value": float(np.sum(dy_v ** 2)), "dy": dy, "dy_key": dy_k, "dy_value": dy_v}
