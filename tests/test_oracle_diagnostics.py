"""Pins for the output-space error oracle (CPU only): "Output-Aware
Rotation for INT2 KV-Cache Quantization" §3.2, Eqs. (5)-(10)."""
import math

import numpy as np

from bit_kv_cache_13_gb300 import inputs
from oracle import diagnostics


def _case(rng, T=30, h_q=6, h_kv=2, d_model=40):
    q = rng.standard_normal((h_q, 128))
    k = rng.standard_normal((T, h_kv, 128)) * 2
    v = rng.standard_normal((T, h_kv, 128))
    w_o = rng.standard_normal((h_q, d_model, 128)) / math.sqrt(128)
    return q, k, v, w_o


def test_key_and_value_terms_add_up_to_the_output_error():
    # Eq. (8) is an identity: sum p~ v~ - sum p v = sum (p~ - p) v + sum p~ (v~ - v).
    rng = np.random.default_rng(51)
    q, k, v, w_o = _case(rng)
    kt = k + 0.3 * rng.standard_normal(k.shape)
    vt = v + 0.2 * rng.standard_normal(v.shape)
    r = diagnostics.output_error(q, k, v, kt, vt, w_o, 1 / math.sqrt(128))
    assert np.max(np.abs(r["dy_key"] + r["dy_value"] - r["dy"])) <= 1e-12 * np.max(np.abs(r["dy"]))
    assert r["E_out"] > 0 and r["E_out_key"] > 0 and r["E_out_value"] > 0


def test_exact_cache_has_no_error():
    rng = np.random.default_rng(52)
    q, k, v, w_o = _case(rng)
    r = diagnostics.output_error(q, k, v, k, v, w_o, 0.1)
    assert r["E_rec"] == 0 and r["E_out"] == 0


def test_value_only_error_has_no_key_term():
    # With exact keys the attention map is unchanged (Delta p = 0), so the
    # whole output error is p (Delta v) W_O^T.
    rng = np.random.default_rng(53)
    q, k, v, w_o = _case(rng)
    dv = 0.1 * rng.standard_normal(v.shape)
    r = diagnostics.output_error(q, k, v, k, v + dv, w_o, 0.1)
    assert r["E_out_key"] == 0
    assert abs(r["E_rec"] - float(np.sum(dv ** 2))) <= 1e-12 * r["E_rec"]
    for j in range(6):
        a = k[:, j // 3] @ q[j] * 0.1
        p = np.exp(a - a.max())
        p /= p.sum()
        want = (p @ dv[:, j // 3]) @ w_o[j].T
        assert np.max(np.abs(r["dy"][j] - want)) <= 1e-12 * np.max(np.abs(want))


def test_reconstruction_error_is_rotation_invariant():
    # Eq. (4): D_R(z) = Q2(zR) R^T; an orthogonal change of basis of the
    # error leaves E_rec unchanged (the Frobenius norm is invariant), while
    # the output error depends on q, the attention map and W_O.
    rng = np.random.default_rng(54)
    q, k, v, w_o = _case(rng)
    ek = 0.2 * rng.standard_normal(k.shape)
    ev = 0.2 * rng.standard_normal(v.shape)
    r_mat = inputs.head_rotation(128, "diag")
    a = diagnostics.output_error(q, k, v, k + ek, v + ev, w_o, 0.1)
    b = diagnostics.output_error(q, k, v, k + ek @ r_mat.T, v + ev @ r_mat.T, w_o, 0.1)
    assert abs(a["E_rec"] - b["E_rec"]) <= 1e-12 * a["E_rec"]
    assert abs(a["E_out"] - b["E_out"]) > 1e-6 * a["E_out"]
