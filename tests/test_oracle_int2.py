"""Pins for the INT2 oracle (CPU only).

Output-Aware Rotation for INT2 KV-Cache Quantization: §1 (INT2 = 1/8 of
BF16, one scale per group, centring keeps the softmax), §3 Eqs. (1)-(2)
(attention), §3.1 Eq. (4) (D_R(z) = Q2(zR)R^T, identity when Q2 is).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from bit_kv_cache_13_gb300 import inputs
from oracle import attention, int2


# ---------------------------------------------------------------- rotations

def test_hadamard_and_rotation_orthogonal():
    h = inputs.sylvester_hadamard(128)
    assert np.array_equal(h @ h.T, 128 * np.eye(128))
    r = inputs.head_rotation(128, "t", 0)
    assert np.max(np.abs(r @ r.T - np.eye(128))) <= 1e-12
    assert np.max(np.abs(r.T @ r - np.eye(128))) <= 1e-12


def test_eq4_identity_when_quantiser_is_identity():
    # D_R(z) = (zR)R^T = z
    r = inputs.head_rotation(128, "t", 1)
    z = np.random.default_rng(0).standard_normal((50, 128)) * 7
    assert np.max(np.abs((z @ r) @ r.T - z)) <= 1e-12 * np.max(np.abs(z))


def test_attention_invariant_under_rotation_and_centring():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 128))
    k = rng.standard_normal((300, 1, 128)) * 3 + rng.standard_normal(128) * 5
    v = rng.standard_normal((300, 1, 128))
    s = 1 / math.sqrt(128)
    base = attention.gqa_decode(q, k, v, s)
    mu = k[:, 0].mean(0)
    cent = attention.gqa_decode(q, k - mu, v, s)
    assert np.max(np.abs(base - cent)) <= 1e-12
    rk, rv = inputs.head_rotation(128, "a"), inputs.head_rotation(128, "b")
    rot = attention.gqa_decode(q @ rk, (k - mu) @ rk, v @ rv, s) @ rv.T
    assert np.max(np.abs(base - rot)) <= 1e-12


def test_attention_textbook_loop():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 8))
    k = rng.standard_normal((5, 1, 8))
    v = rng.standard_normal((5, 1, 8))
    got = attention.gqa_decode(q, k, v, 0.5)
    for j in range(2):
        a = [sum(q[j, i] * k[s, 0, i] for i in range(8)) * 0.5 for s in range(5)]
        e = [math.exp(x) for x in a]
        tot = sum(e)
        for i in range(8):
            want = sum(e[s] / tot * v[s, 0, i] for s in range(5))
            assert abs(got[j, i] - want) <= 1e-13


# ---------------------------------------------------------------- quantiser

def _brute_codes(x32, scale_h, min_h):
    """Exact nearest level by rational distances; ties to the lower code."""
    out = []
    sc, mn = Fraction(float(scale_h)), Fraction(float(min_h))
    for x in x32:
        xf = Fraction(float(x))
        if sc == 0:
            out.append(0)
            continue
        d = [abs(xf - (mn + c * sc)) for c in range(4)]
        out.append(int(min(range(4), key=lambda c: (d[c], c))))
    return np.array(out)


def test_codes_are_nearest_level_random():
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(0.01, 50) + rng.normal(0, 20)).astype(np.float32)
        sc, mn = int2.quant_params(x)
        got = int2.quant_codes(x, sc, mn)
        assert np.array_equal(got, _brute_codes(x, sc, mn))


def test_codes_midpoint_ties_go_low():
    # exact midpoints between levels: min = 1, scale = 0.5, x = 1.25, 1.75, 2.25
    sc, mn = np.float16(0.5), np.float16(1.0)
    x = np.array([1.0, 1.25, 1.5, 1.75, 2.0, 2.25, 2.5, 2.5000002, 1.2499999], np.float32)
    got = int2.quant_codes(x, sc, mn)
    assert got.tolist() == [0, 0, 1, 1, 2, 2, 3, 3, 0]
    assert np.array_equal(got, _brute_codes(x, sc, mn))


def test_quant_params_cover_range():
    rng = np.random.default_rng(5)
    for _ in range(300):
        x = (rng.standard_normal(32) * rng.uniform(1e-3, 100)).astype(np.float32)
        sc, mn = int2.quant_params(x)
        codes = int2.quant_codes(x, sc, mn)
        xh = int2.dequantize(np.tile(codes, 4), np.full(4, sc), np.full(4, mn))[:32]
        lo, hi = float(x.min()), float(x.max())
        slack = abs(float(mn) - lo) + 3 * abs(float(sc) - (hi - lo) / 3)
        assert np.max(np.abs(xh - x)) <= (hi - lo) / 6 + slack + 1e-12
        assert 0 <= codes.min() and codes.max() <= 3


def test_constant_group_scale_zero():
    x = np.full(32, 3.140625, np.float32)
    sc, mn = int2.quant_params(x)
    assert float(sc) == 0.0 and float(mn) == 3.140625
    assert int2.quant_codes(x, sc, mn).max() == 0


def test_scale_underflow_and_overflow_saturate():
    x = np.zeros(32, np.float32)
    x[1] = 1e-9
    sc, mn = int2.quant_params(x)
    assert float(sc) == 0.0
    x = np.zeros(32, np.float32)
    x[0], x[1] = -1e6, 1e6
    sc, mn = int2.quant_params(x)
    assert float(sc) == 65504.0 and float(mn) == -65504.0


def test_storage_is_one_eighth_of_bf16():
    acc = int2.storage_bytes_per_token_head()
    assert acc["k_codes"] * 8 == int2.D * 2            # 2 bits vs 16 bits
    assert acc["total"] == 96 and acc["bf16_kv"] == 512
    assert int2.TILE_BYTES == int2.PAGE * acc["total"]


def test_pack_layout_and_roundtrip():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 4, size=(10, 128)).astype(np.uint8)
    assert np.array_equal(int2.unpack_codes(int2.pack_codes(codes)), codes)
    one = np.zeros(128, np.uint8)
    one[32 * 2 + 4 * 5 + 3] = 2               # group 2, byte-row 5, position 3
    rec = int2.pack_codes(one)
    assert rec.tolist() == [0] * (4 * 5 + 2) + [2 << 6] + [0] * (32 - 4 * 5 - 3)
    sc = np.array([1.5, 0.0, 65504.0, 2.0 ** -24], np.float16)
    mn = np.array([-2.0, 3.0, -65504.0, 0.5], np.float16)
    raw = int2.pack_meta(sc, mn)
    assert raw.shape == (16,)
    s2, m2 = int2.unpack_meta(raw)
    assert np.array_equal(s2, sc) and np.array_equal(m2, mn)


def test_meta_placement_covers_the_tile():
    """Key meta: one 16-byte record per slot; value meta: pair-major words
    (scales of slots 2j, 2j+1 of one group, then the same for the mins)."""
    for side, lo in ((0, int2.OFF_K_META), (1, int2.OFF_V_META)):
        allb = np.concatenate([int2.meta_bytes(side, s) for s in range(int2.PAGE)])
        assert sorted(allb.tolist()) == list(range(lo, lo + 256))
    assert int2.meta_bytes(0, 3).tolist() == list(range(512 + 48, 512 + 64))
    # slot 3 = pair 1, upper half; group 2: scale bytes 1280 + 16 + 8 + 2, min bytes 128 further
    assert int2.meta_bytes(1, 3)[8:12].tolist() == [1306, 1307, 1434, 1435]
    assert int2.meta_bytes(1, 0)[:4].tolist() == [1280, 1281, 1408, 1409]
    # a tile written by append: slot 5's value scales sit in the pair-2 words
    cache = int2.new_cache(1, 1)
    w = np.zeros((6, 1, 128), np.float32)
    w[5, 0, :32] = np.linspace(0.0, 3.0, 32)         # group 0: min 0, scale 1
    int2.append(cache, np.zeros_like(w), w, np.arange(6), np.zeros((1, 128), np.float32),
                np.eye(128, dtype=np.float32)[None], np.eye(128, dtype=np.float32)[None])
    word = cache[0, 0, 1280 + 16 * 2: 1280 + 16 * 2 + 4].view(np.float16)
    assert word.tolist() == [0.0, 1.0]                 # (slot 4, slot 5) scales of group 0


# ---------------------------------------------------------------- end to end

def _lattice_keys(rng, n, mu, r):
    """Keys whose centred rotations sit exactly on INT2 levels (fp16 min and
    scale, min and max both present), so Q2 is the identity on them."""
    z = np.zeros((n, 128))
    for t in range(n):
        for g in range(4):
            m = float(np.float16(rng.uniform(-4, 4)))
            s = float(np.float16(rng.uniform(0.25, 2)))
            c = rng.integers(0, 4, 32)
            c[0], c[1] = 0, 3
            z[t, 32 * g: 32 * g + 32] = m + s * c
    return z @ r.T + mu, z


def test_decode_reduces_to_plain_attention_on_lattice_inputs():
    rng = np.random.default_rng(8)
    h_kv, g, T = 2, 3, 40
    rk = np.stack([inputs.head_rotation(128, "k", h) for h in range(h_kv)]).astype(np.float32)
    rv = np.stack([inputs.head_rotation(128, "v", h) for h in range(h_kv)]).astype(np.float32)
    mu = (rng.standard_normal((h_kv, 128)) * 3).astype(np.float32)
    k = np.zeros((T, h_kv, 128))
    v = np.zeros((T, h_kv, 128))
    for h in range(h_kv):
        k[:, h], _ = _lattice_keys(rng, T, mu[h].astype(np.float64), rk[h].astype(np.float64))
        v[:, h], _ = _lattice_keys(rng, T, 0.0, rv[h].astype(np.float64))
    k = k.astype(np.float32)
    v = v.astype(np.float32)
    cache = int2.new_cache(8, h_kv)
    bt = np.array([[5, 2, 7]], np.int32)
    slots = np.array([bt[0, t // 16] * 16 + t % 16 for t in range(T)])
    int2.append(cache, k, v, slots, mu, rk, rv)
    q = rng.standard_normal((1, h_kv * g, 128))
    got = int2.decode(q, cache, bt, [T], mu, rk, rv, 1 / math.sqrt(128), h_kv)
    want = attention.gqa_decode(q[0], k.astype(np.float64), v.astype(np.float64), float(np.float32(1 / math.sqrt(128))))
    assert np.max(np.abs(got[0] - want)) <= 1e-4 * np.max(np.abs(want))


def test_decode_kivi_special_case_matches_dense_loop():
    # R = I, mu = 0: plain per-token group quantisation, then the textbook
    # softmax over explicitly dequantised keys and values.
    rng = np.random.default_rng(10)
    T = 21
    k = (rng.standard_normal((T, 1, 128)) * 2).astype(np.float32)
    v = rng.standard_normal((T, 1, 128)).astype(np.float32)
    eye = np.eye(128, dtype=np.float32)[None]
    mu = np.zeros((1, 128), np.float32)
    cache = int2.new_cache(2, 1)
    int2.append(cache, k, v, np.arange(T), mu, eye, eye)
    q = rng.standard_normal((1, 2, 128))
    got = int2.decode(q, cache, np.array([[0, 1]]), [T], mu, eye, eye, 0.125, 1)
    kq = np.zeros((T, 128))
    vq = np.zeros((T, 128))
    for t in range(T):
        for src, dst in ((k, kq), (v, vq)):
            for gi in range(4):
                grp = src[t, 0, 32 * gi: 32 * gi + 32]
                lo, hi = float(grp.min()), float(grp.max())
                sc = float(np.float16(np.float32(np.float32(hi - lo) / np.float32(3))))
                mn = float(np.float16(lo))
                for i in range(32):
                    levels = [mn + c * sc for c in range(4)]
                    dist = [abs(float(grp[i]) - L) for L in levels]
                    c = 0 if sc == 0 else min(range(4), key=lambda c: (dist[c], c))
                    dst[t, 32 * gi + i] = levels[c]
    for j in range(2):
        a = [float(kq[s] @ q[0, j]) * 0.125 for s in range(T)]
        m = max(a)
        e = [math.exp(x - m) for x in a]
        want = sum(e[s] * vq[s] for s in range(T)) / sum(e)
        assert np.max(np.abs(got[0, j] - want)) <= 1e-12 * np.max(np.abs(want)) + 1e-13


def test_decode_page_order_is_logical():
    rng = np.random.default_rng(11)
    T = 37
    k = rng.standard_normal((T, 1, 128)).astype(np.float32)
    v = rng.standard_normal((T, 1, 128)).astype(np.float32)
    rk = inputs.head_rotation(128, "x").astype(np.float32)[None]
    mu = np.zeros((1, 128), np.float32)
    q = rng.standard_normal((1, 4, 128))
    outs = []
    for table in ([0, 1, 2], [9, 4, 6]):
        cache = int2.new_cache(10, 1)
        slots = [table[t // 16] * 16 + t % 16 for t in range(T)]
        int2.append(cache, k, v, slots, mu, rk, rk)
        outs.append(int2.decode(q, cache, np.array([table]), [T], mu, rk, rk, 0.1, 1))
    assert np.array_equal(outs[0], outs[1])


def test_empty_context_gives_zeros():
    cache = int2.new_cache(1, 1)
    eye = np.eye(128, dtype=np.float32)[None]
    out = int2.decode(np.ones((1, 4, 128)), cache, np.array([[0]]), [0], np.zeros((1, 128)), eye, eye, 0.1, 1)
    assert np.all(out == 0)


def test_seventy_b_kv_byte_count():
    # RoPE-aware allocation page, motivation: 80 layers x 8 KV heads x 128
    # dims x (K, V) x fp16 = 320 KiB per token, ~40 GiB at 128K tokens.
    per_token = 80 * 8 * 128 * 2 * 2
    assert per_token == 320 * 1024
    assert per_token * 131072 == 40 * 1024 ** 3


# ---------------------------------------------------------------- BF16 window

def _lattice_tokens_identity(rng, T, mu):
    """Tokens k = z + mu (R = I) whose 32-channel groups are exactly the four
    INT2 levels m + c*s of their own min/max, so the INT2 round trip is
    exact; every value is a small multiple of 1/4, exact in bf16 and fp32."""
    z = np.zeros((T, 128))
    for t in range(T):
        for g in range(4):
            m = 0.25 * rng.integers(-8, 8)
            s = 0.25 * rng.integers(1, 5)
            c = rng.integers(0, 4, 32)
            c[0], c[1] = 0, 3
            z[t, 32 * g: 32 * g + 32] = m + s * c
    return z + mu


def _split_window(k, v, w):
    """The last w tokens as a one-sequence window [1, w, H_kv, d]."""
    T = k.shape[0]
    return k[:T - w], v[:T - w], (k[None, T - w:], v[None, T - w:], [w])


def test_window_token_equals_exact_int2_token():
    # A token whose INT2 encoding is exact (R = I, lattice groups) attends
    # the same from the packed cache as from the BF16 window, so moving the
    # last w tokens into the window leaves the output unchanged.
    rng = np.random.default_rng(21)
    T, w, g = 35, 6, 4
    mu = (0.25 * rng.integers(-8, 8, (1, 128))).astype(np.float32)
    k = _lattice_tokens_identity(rng, T, mu[0].astype(np.float64))[:, None].astype(np.float32)
    v = _lattice_tokens_identity(rng, T, 0.0)[:, None].astype(np.float32)
    eye = np.eye(128, dtype=np.float32)[None]
    q = rng.standard_normal((1, g, 128))
    full = int2.new_cache(3, 1)
    int2.append(full, k, v, np.arange(T), mu, eye, eye)
    want = int2.decode(q, full, np.array([[0, 1, 2]]), [T], mu, eye, eye, 0.125, 1)
    kh, vh, win = _split_window(k, v, w)
    part = int2.new_cache(3, 1)
    int2.append(part, kh, vh, np.arange(T - w), mu, eye, eye)
    got = int2.decode(q, part, np.array([[0, 1, 2]]), [T - w], mu, eye, eye, 0.125, 1, window=win)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_window_token_matches_rotated_lattice_token():
    # Same move with a Haar-Hadamard R and a non-zero centre: the cached keys
    # are lattice points in the rotated basis, so the window and the cache
    # agree to the fp32 rounding of k = z R^T + mu.
    rng = np.random.default_rng(22)
    T, w, g = 40, 9, 3
    rk = inputs.head_rotation(128, "k", 0).astype(np.float32)[None]
    rv = inputs.head_rotation(128, "v", 0).astype(np.float32)[None]
    mu = (rng.standard_normal((1, 128)) * 3).astype(np.float32)
    k, _ = _lattice_keys(rng, T, mu[0].astype(np.float64), rk[0].astype(np.float64))
    v, _ = _lattice_keys(rng, T, 0.0, rv[0].astype(np.float64))
    k = k[:, None].astype(np.float32)
    v = v[:, None].astype(np.float32)
    q = rng.standard_normal((1, g, 128))
    bt = np.array([[4, 1, 3]], np.int32)
    slots = lambda n: np.array([bt[0, t // 16] * 16 + t % 16 for t in range(n)])
    full = int2.new_cache(6, 1)
    int2.append(full, k, v, slots(T), mu, rk, rv)
    want = int2.decode(q, full, bt, [T], mu, rk, rv, 1 / math.sqrt(128), 1)
    kh, vh, win = _split_window(k, v, w)
    part = int2.new_cache(6, 1)
    int2.append(part, kh, vh, slots(T - w), mu, rk, rv)
    got = int2.decode(q, part, bt, [T - w], mu, rk, rv, 1 / math.sqrt(128), 1, window=win)
    assert np.max(np.abs(got - want)) <= 1e-4 * np.max(np.abs(want))


def test_window_alone_is_plain_attention():
    # No cached tokens: the output is textbook attention over the window.
    rng = np.random.default_rng(23)
    W, h_kv, g = 7, 2, 4
    kw = rng.standard_normal((1, W, h_kv, 128)).astype(np.float32)
    vw = rng.standard_normal((1, W, h_kv, 128)).astype(np.float32)
    eye = np.stack([np.eye(128, dtype=np.float32)] * h_kv)
    q = rng.standard_normal((1, h_kv * g, 128))
    cache = int2.new_cache(1, h_kv)
    got = int2.decode(q, cache, np.array([[0]]), [0], np.zeros((h_kv, 128)), eye, eye, 0.1, h_kv,
                      window=(kw, vw, [W]))
    for j in range(h_kv * g):
        a = kw[0, :, j // g].astype(np.float64) @ q[0, j] * float(np.float32(0.1))
        e = np.exp(a - a.max())
        want = (e[:, None] * vw[0, :, j // g]).sum(0) / e.sum()
        assert np.max(np.abs(got[0, j] - want)) <= 1e-12 * np.max(np.abs(want))


def test_window_lengths_are_per_sequence():
    # Ragged windows: sequence b attends exactly its first win_lens[b] window
    # tokens (zero-length windows included); entries past that are ignored.
    rng = np.random.default_rng(24)
    B, W, T = 3, 5, 20
    k = rng.standard_normal((B, T, 1, 128)).astype(np.float32)
    v = rng.standard_normal((B, T, 1, 128)).astype(np.float32)
    kw = rng.standard_normal((B, W, 1, 128)).astype(np.float32)
    vw = rng.standard_normal((B, W, 1, 128)).astype(np.float32)
    rk = inputs.head_rotation(128, "w").astype(np.float32)[None]
    mu = np.zeros((1, 128), np.float32)
    q = rng.standard_normal((B, 2, 128))
    cache = int2.new_cache(2 * B, 1)
    bt = np.array([[2 * b, 2 * b + 1] for b in range(B)], np.int32)
    for b in range(B):
        int2.append(cache, k[b], v[b], [bt[b, t // 16] * 16 + t % 16 for t in range(T)], mu, rk, rk)
    lens = [0, 3, 5]
    got = int2.decode(q, cache, bt, [T] * B, mu, rk, rk, 0.1, 1, window=(kw, vw, lens))
    for b in range(B):
        poisoned = kw.copy()
        poisoned[b, lens[b]:] = 1e4                      # beyond the length: must not matter
        one = int2.decode(q[b:b + 1], cache, bt[b:b + 1], [T], mu, rk, rk, 0.1, 1,
                          window=(poisoned[b:b + 1], vw[b:b + 1], [lens[b]]))
        assert np.array_equal(got[b], one[0])
        if lens[b] == 0:
            plain = int2.decode(q[b:b + 1], cache, bt[b:b + 1], [T], mu, rk, rk, 0.1, 1)
            assert np.array_equal(got[b], plain[0])


# ---------------------------------------------------------------- clip ratio

def test_clip_one_is_the_plain_range():
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((50, 4, 32)) * 3 + 1).astype(np.float32)
    for a, b in zip(int2.quant_params(x), int2.quant_params(x, 1.0)):
        assert np.array_equal(a, b)


def test_clipped_codes_are_the_nearest_level():
    # With c < 1 the four levels span [c*min, c*max] (to fp16 rounding) and
    # every value takes the nearest of them, ties low: values beyond the
    # clipped range saturate at code 0 or 3.
    rng = np.random.default_rng(42)
    for c in (0.5, 0.8, 0.95):
        for _ in range(100):
            x = (rng.standard_normal(32) * rng.uniform(0.1, 20) + rng.normal(0, 5)).astype(np.float32)
            sc, mn = int2.quant_params(x, c)
            lo = float(np.float32(np.float32(c) * x.min()))
            hi = float(np.float32(np.float32(c) * x.max()))
            assert float(mn) == float(np.float16(lo))
            assert abs(float(mn) + 3 * float(sc) - hi) <= 2e-3 * max(abs(hi), abs(lo)) + 1e-6
            got = int2.quant_codes(x, sc, mn)
            assert np.array_equal(got, _brute_codes(x, sc, mn))
            if float(sc) > 0:
                assert np.all(got[x >= hi] == 3) and np.all(got[x <= lo] == 0)


def test_clipping_lowers_the_error_of_heavy_tailed_groups():
    # Student-t (3 dof) groups: a few large values stretch the plain range;
    # a clip ratio somewhat below 1 gives a lower mean squared error.
    rng = np.random.default_rng(43)
    x = rng.standard_t(3, size=(4000, 4, 32)).astype(np.float32)
    def mse(c):
        codes, sc, mn = int2.quantize(x.reshape(4000, 128), c)
        return float(np.mean((int2.dequantize(codes, sc, mn) - x.reshape(4000, 128)) ** 2))
    assert mse(0.8) < 0.95 * mse(1.0)


def test_dequantize_f32_is_the_rounded_fp64_value():
    rng = np.random.default_rng(44)
    z = (rng.standard_normal((20, 128)) * 5).astype(np.float32)
    codes, sc, mn = int2.quantize(z)
    d32 = int2.dequantize_f32(codes, sc, mn)
    assert d32.dtype == np.float32
    assert np.array_equal(d32, int2.dequantize(codes, sc, mn).astype(np.float32))
