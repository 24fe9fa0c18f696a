"""Pins for the Block-GTQ oracle (CPU only).

RoPE-Aware Bit Allocation for KV-Cache Quantization: prerequisites (RoPE
block structure, TQ-MSE and its 4^-b error law, greedy allocation and
Theorem 1), core method (logit block decomposition, key-error logit bound),
method steps (3)-(4) (grouped encoding, uniform values).
"""
import itertools
import math

import numpy as np
import pytest
import torch
from scipy import integrate

from bit_kv_cache_13_gb300 import inputs
from oracle import attention, bgtq

# Max (1960) / Lloyd (1982) Gaussian quantiser tables, positive half; the
# tabulated MSEs carry four significant digits of the original tables.
TEXTBOOK_LEVELS = {
    2: [0.4528, 1.5104],
    3: [0.2451, 0.7560, 1.3440, 2.1520],
}
TEXTBOOK_MSE = {1: 0.3634, 2: 0.1175, 3: 0.03454, 4: 0.009497}


@pytest.fixture(scope="module")
def table():
    return bgtq.lloyd_max_table()


def _mse(c):
    t = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
    tot = 0.0
    for i, ci in enumerate(c):
        tot += integrate.quad(lambda x: (x - ci) ** 2 * math.exp(-x * x / 2) / math.sqrt(2 * math.pi),
                              t[i], t[i + 1], epsabs=1e-13, epsrel=1e-12)[0]
    return tot


def test_lloyd_max_b1_closed_form(table):
    c = table[0, :2]
    assert abs(c[1] - math.sqrt(2 / math.pi)) <= 1e-14 and abs(c[0] + math.sqrt(2 / math.pi)) <= 1e-14


@pytest.mark.parametrize("b", [2, 3])
def test_lloyd_max_textbook_levels(table, b):
    c = table[b - 1, : 2 ** b]
    assert np.allclose(c[2 ** (b - 1):], TEXTBOOK_LEVELS[b], atol=1.5e-4)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_lloyd_max_textbook_mse(table, b):
    assert abs(_mse(table[b - 1, : 2 ** b]) - TEXTBOOK_MSE[b]) <= 1e-3 * TEXTBOOK_MSE[b]


@pytest.mark.parametrize("b", range(1, 9))
def test_lloyd_max_fixed_point_by_quadrature(table, b):
    # centroid condition checked with numerical integration, independent of
    # the closed-form conditional mean used by the iteration
    c = table[b - 1, : 2 ** b]
    assert np.all(np.diff(c) > 0) and np.allclose(c, -c[::-1], atol=1e-12)
    t = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
    f = lambda x: math.exp(-x * x / 2)
    for i in list(range(min(4, len(c)))) + [len(c) // 2, len(c) - 1]:
        m0 = integrate.quad(f, t[i], t[i + 1], epsabs=1e-15, epsrel=1e-13)[0]
        m1 = integrate.quad(lambda x: x * f(x), t[i], t[i + 1], epsabs=1e-15, epsrel=1e-13)[0]
        assert abs(m1 / m0 - c[i]) <= 1e-8


def test_lloyd_max_high_rate_constant(table):
    # Panter-Dite: MSE_b * 4^b rises towards sqrt(3)*pi/2 from below; this is
    # the constant of the TQ-MSE error law
    r = [_mse(table[b - 1, : 2 ** b]) * 4.0 ** b for b in (4, 6, 8)]
    assert r[0] < r[1] < r[2] < bgtq.C_TQ and r[2] > 0.98 * bgtq.C_TQ
    assert abs(bgtq.C_TQ - 2.7207) < 1e-4


def test_greedy_is_optimal_by_brute_force():
    # Theorem 1: greedy minimises J(b) = sum s_i 4^-b_i over integer widths
    rng = np.random.default_rng(0)
    for L in range(1, 6):
        for _ in range(12):
            s = rng.lognormal(0, 2, L)
            for total in range(L, 4 * L + 1):
                w = bgtq.greedy_allocate(s, 1, 4, total)
                assert w.sum() == total and w.min() >= 1 and w.max() <= 4
                best = min(bgtq.objective(s, c) for c in itertools.product(range(1, 5), repeat=L)
                           if sum(c) == total)
                assert bgtq.objective(s, w) <= best * (1 + 1e-12)


def test_greedy_ties_lowest_index_and_cap():
    w = bgtq.greedy_allocate([1.0, 1.0, 1.0], 1, 8, 4)
    assert w.tolist() == [2, 1, 1]
    w = bgtq.greedy_allocate([4.0, 1.0], 1, 8, 3)     # 4*4^-1 == 1*4^0: tie
    assert w.tolist() == [2, 1]
    w = bgtq.greedy_allocate([100.0, 1.0], 1, 3, 100)  # budget above L*b_max
    assert w.tolist() == [3, 3]


def test_greedy_budget_at_config_scale():
    s = inputs.block_energies(inputs.SPECS["bgtq"], 0, 3)
    w = bgtq.greedy_allocate(s, 1, 8, 192)
    assert w.sum() == 192 and w.min() >= 1 and w.max() <= 8
    # more energy never gets fewer bits
    order = np.argsort(-s, kind="stable")
    assert np.all(np.diff(w[order]) <= 0)


def test_pack_bits_lsb_first():
    st = bgtq.pack_bits([1, 2, 5], [1, 2, 3], 1)
    # value 1 (1 bit) -> bit0; value 2 (2 bits) -> bits1..2 = 0,1; 5 (3 bits) -> bits 3..5 = 1,0,1
    assert st.tolist() == [0b101101]
    rng = np.random.default_rng(3)
    widths = rng.integers(1, 9, 70)
    vals = [int(rng.integers(0, 2 ** w)) for w in widths]
    nb = (int(widths.sum()) + 7) // 8
    assert bgtq.unpack_bits(bgtq.pack_bits(vals, widths, nb), widths).tolist() == vals


def test_tile_layout_sizes():
    lay = bgtq.tile_layout(192, 3)
    assert lay["kb"] == 48 and lay["vb"] == 48
    assert lay["tile"] == 16 * (48 + 16 + 48 + 2) and lay["tile"] % 16 == 0


@pytest.mark.parametrize("n", [2, 8, 32, 128])
def test_tq_mse_error_law(table, n):
    # E||x - x^||^2 <= ||x||^2 * C_TQ * 4^-b with C_TQ = sqrt(3)*pi/2,
    # Monte-Carlo with a 3-standard-error margin, vectors of mixed norm
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(n)
    m = 4000 if n <= 32 else 1500
    x = (rng.standard_normal((m, n)) * rng.lognormal(0, 1, (m, 1))).astype(np.float32)
    for b in (1, 2, 3, 4, 6):
        cb = bgtq.scaled_codebook(table, b, n)
        codes, nh, r, _ = bgtq.tq_encode(x, pis[n], cb)
        xh = bgtq.tq_decode(codes, nh, pis[n], cb)
        rel = np.sum((xh - x) ** 2, -1) / np.sum(x.astype(np.float64) ** 2, -1)
        mean = rel.mean() + 3 * rel.std() / math.sqrt(m)
        assert mean <= bgtq.C_TQ * 4.0 ** -b, (n, b, mean)


def test_tq_norm_and_zero_vector(table):
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    x = np.zeros((2, 8), np.float32)
    x[1, 3] = 5.0
    codes, nh, r, y = bgtq.tq_encode(x, pis[8], bgtq.scaled_codebook(table, 3, 8))
    assert codes[0].max() == 0 and float(nh[0]) == 0.0
    assert float(r[1]) == 5.0 and float(nh[1]) == 5.0
    assert abs(np.sum(y[1].astype(np.float64) ** 2) - 1) <= 1e-6


def test_rope_block_decomposition_and_relative_position():
    rng = np.random.default_rng(5)
    q = torch.tensor(rng.standard_normal((1, 128)), dtype=torch.float64)
    k = torch.tensor(rng.standard_normal((1, 128)), dtype=torch.float64)
    vals = []
    for m, n in ((10, 3), (1010, 1003), (77, 70)):
        qm = inputs.rope_apply(q, torch.tensor([m]), 5e5)
        kn = inputs.rope_apply(k, torch.tensor([n]), 5e5)
        vals.append(float((qm * kn).sum()))
        blocks = sum(float(qm[0, i] * kn[0, i] + qm[0, i + 64] * kn[0, i + 64]) for i in range(64))
        assert abs(blocks - vals[-1]) <= 1e-12 * abs(vals[-1]) + 1e-12
    assert abs(vals[0] - vals[1]) <= 1e-9 and abs(vals[0] - vals[2]) <= 1e-9


def test_key_error_logit_bound(table):
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(12)
    s = rng.lognormal(0, 2, 64)
    w = bgtq.greedy_allocate(s, 1, 8, 192)
    sd = np.sqrt(np.concatenate([s, s]) / 2)
    for _ in range(30):
        k = (rng.standard_normal(128) * sd).astype(np.float32)
        q = rng.standard_normal(128) * sd
        kh = np.zeros(128)
        for b, bl in bgtq.width_groups(w):
            if not bl:
                continue
            n = 2 * len(bl)
            cb = bgtq.scaled_codebook(table, b, n)
            codes, nh, _, _ = bgtq.tq_encode(bgtq.gather(k, bl), pis[n], cb)
            bgtq.scatter(bgtq.tq_decode(codes, nh, pis[n], cb), bl, kh)
        e = kh - k.astype(np.float64)
        bound = sum(math.hypot(q[i], q[i + 64]) * math.hypot(e[i], e[i + 64]) for i in range(64))
        assert abs(q @ kh - q @ k) <= bound * (1 + 1e-12)


def test_decode_close_to_plain_attention_at_high_width(table):
    # with 8-bit keys and values the packed-cache decode approaches the
    # unquantised attention; a transposed rotation would not
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(13)
    T, h_kv = 20, 1
    k = rng.standard_normal((T, h_kv, 128)).astype(np.float32)
    v = rng.standard_normal((T, h_kv, 128)).astype(np.float32)
    widths = np.full((h_kv, 64), 8)
    total = 8 * 64
    cache = bgtq.new_cache(2, h_kv, total, 8)
    bgtq.append(cache, k, v, np.arange(T), widths, 8, total, pis, table)
    q = rng.standard_normal((1, 2, 128))
    got = bgtq.decode(q, cache, np.array([[0, 1]]), [T], widths, 8, total, pis, table, 0.1, h_kv)
    want = attention.gqa_decode(q[0], k, v, float(np.float32(0.1)))
    assert np.max(np.abs(got[0] - want)) <= 0.02 * np.max(np.abs(want))


# ------------------------------------------------------ calibration energy scores

def test_energy_scores_hand_example():
    # d = 4: block 0 = dims (0, 2), block 1 = dims (1, 3); two tokens, two
    # query heads on one KV head.
    q = np.array([[[1, 2, 2, 0], [0, 0, 3, 4]],
                  [[3, 0, 4, 1], [1, 1, 1, 1]]], dtype=np.float64)      # [T=2, H_q=2, 4]
    k = np.array([[[2, 0, 0, 1]], [[0, 3, 4, 0]]], dtype=np.float64)    # [T=2, H_kv=1, 4]
    s, s_star = bgtq.energy_scores(q, k, 1)
    # ||q(0)||^2: t0 = (1, 2)->5, (0, 3)->9; t1 = (3, 4)->25, (1, 1)->2 -> mean 41/4
    # ||q(1)||^2: t0 = (2, 0)->4, (0, 4)->16; t1 = (0, 1)->1, (1, 1)->2 -> mean 23/4
    # ||k(0)||^2: t0 = (2, 0)->4; t1 = (0, 4)->16 -> mean 10;  ||k(1)||^2: 1, 9 -> mean 5
    assert np.allclose(s, [[0.5 * 41 / 4 + 0.5 * 10, 0.5 * 23 / 4 + 0.5 * 5]], rtol=0, atol=1e-15)
    pairs0 = [math.sqrt(5) * 2, 3 * 2, 5 * 4, math.sqrt(2) * 4]
    pairs1 = [2 * 1, 4 * 1, 1 * 3, math.sqrt(2) * 3]
    assert np.allclose(s_star, [[sum(pairs0) / 4, sum(pairs1) / 4]], rtol=1e-15, atol=0)


def test_energy_scores_am_gm_bound():
    rng = np.random.default_rng(31)
    q = rng.standard_normal((200, 8, 128)) * rng.lognormal(0, 1.5, 128)
    k = rng.standard_normal((200, 2, 128)) * rng.lognormal(0, 1.5, 128)
    s, s_star = bgtq.energy_scores(q, k, 2)
    assert np.all(s_star <= s * (1 + 1e-15))
    assert np.any(s_star < 0.9 * s)                   # the bound is not tight in general


def test_energy_scores_equal_when_queries_are_the_keys():
    # AM-GM holds with equality when ||q(i)|| = ||k(i)|| token by token.
    rng = np.random.default_rng(32)
    k = rng.standard_normal((50, 3, 128))
    s, s_star = bgtq.energy_scores(k.copy(), k, 3)
    assert np.allclose(s_star, s, rtol=1e-14, atol=0)
    assert np.allclose(s, ((k[..., :64] ** 2 + k[..., 64:] ** 2)).mean(axis=0), rtol=1e-14, atol=0)


def test_energy_scores_invariant_under_rope():
    # Rotate-half RoPE turns block i = dims (i, i + 64) by a 2x2 rotation,
    # which keeps every block norm: scores from pre- and post-RoPE vectors
    # agree (a wrong pairing of dims would break this).
    rng = np.random.default_rng(33)
    T = 64
    q = torch.as_tensor(rng.standard_normal((T, 4, 128)))
    k = torch.as_tensor(rng.standard_normal((T, 1, 128)) * 3)
    pos = torch.as_tensor(rng.integers(0, 100000, T))
    qr = torch.stack([inputs.rope_apply(q[:, j], pos, 5e5) for j in range(4)], dim=1)
    kr = inputs.rope_apply(k[:, 0], pos, 5e5)[:, None]
    a = bgtq.energy_scores(q.numpy(), k.numpy(), 1)
    b = bgtq.energy_scores(qr.numpy(), kr.numpy(), 1)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-12, atol=0)


def test_energy_scores_recover_the_generators_block_energies():
    # The Block-GTQ workload draws q and k block i with E||.(i)||^2 = s_i;
    # 4096 calibration tokens recover every s_i to well within 10 % (the
    # relative standard error is about 1/sqrt(T) = 1.6 %).
    spec = inputs.small_spec("cal", h_q=8, h_kv=2, batch=1, ctx=4096, k_kind="energy_rope")
    pos = torch.arange(4096)
    q = inputs.gen_prefix_queries(spec, 0, pos).float().numpy()
    k = inputs.gen_keys(spec, 0, 0, pos).float().numpy()
    s, _ = bgtq.energy_scores(q, k, 2)
    for h in range(2):
        want = inputs.block_energies(spec, 0, h)
        assert np.max(np.abs(s[h] / want - 1)) < 0.1


# ------------------------------------------------- nearest centroid (tie rule)

def _brute_nearest(y32, cb32):
    """Nearest centroid by exact rational distances; equal distances go to
    the lower index (the reading of the TQ-MSE scalar quantiser taken here)."""
    from fractions import Fraction
    cs = [Fraction(float(c)) for c in np.asarray(cb32, np.float32)]
    out = []
    for y in np.asarray(y32, np.float32).ravel():
        yf = Fraction(float(y))
        d = [abs(yf - c) for c in cs]
        out.append(min(range(len(cs)), key=lambda k: (d[k], k)))
    return np.asarray(out).reshape(np.shape(y32))


@pytest.mark.parametrize("b,n", [(1, 2), (2, 8), (3, 30), (4, 64), (6, 128), (8, 2)])
def test_nearest_codes_brute_force_random(table, b, n):
    cb = bgtq.scaled_codebook(table, b, n)
    rng = np.random.default_rng(100 * b + n)
    y = (rng.standard_normal(400) * 1.3 / np.sqrt(n)).astype(np.float32)
    assert np.array_equal(bgtq.nearest_codes(y, cb), _brute_nearest(y, cb))


def test_nearest_codes_exact_midpoints_go_low():
    # a codebook whose midpoints are exact in fp32: -1, 0, 1 lie exactly
    # between two centroids and must take the lower index; the fp32
    # neighbours on either side go to the nearer centroid
    cb = np.array([-1.5, -0.5, 0.5, 1.5], np.float32)
    mids = np.array([-1.0, 0.0, 1.0], np.float32)
    assert bgtq.nearest_codes(mids, cb).tolist() == [0, 1, 2]
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    assert bgtq.nearest_codes(up, cb).tolist() == [1, 2, 3]
    assert bgtq.nearest_codes(dn, cb).tolist() == [0, 1, 2]
    ends = np.array([-1e30, 1e30, -1.5, 1.5], np.float32)
    assert bgtq.nearest_codes(ends, cb).tolist() == [0, 3, 0, 3]
    allv = np.concatenate([mids, up, dn, ends])
    assert np.array_equal(bgtq.nearest_codes(allv, cb), _brute_nearest(allv, cb))


def test_nearest_codes_ties_on_the_real_codebooks(table):
    # wherever the fp64 midpoint of two adjacent scaled centroids is itself
    # an fp32 value, y on it takes the lower index (brute force agrees); the
    # next fp32 values above it take the upper one
    seen = 0
    for b in range(1, 9):
        for n in (2, 6, 16, 40, 128):
            cb = bgtq.scaled_codebook(table, b, n)
            c64 = cb.astype(np.float64)
            m = 0.5 * (c64[:-1] + c64[1:])
            exact = m.astype(np.float32).astype(np.float64) == m
            if not exact.any():
                continue
            k = np.nonzero(exact)[0]
            y = m[k].astype(np.float32)
            assert np.array_equal(bgtq.nearest_codes(y, cb), k)
            assert np.array_equal(bgtq.nearest_codes(np.nextafter(y, np.float32(np.inf)), cb), k + 1)
            assert np.array_equal(bgtq.nearest_codes(y, cb), _brute_nearest(y, cb))
            seen += len(k)
    assert seen >= 8   # the symmetric codebooks put an exact midpoint at 0 for every width


# ------------------------------------ TQ-MSE with the rotation taken in fp64

def _signed_permutation(n, seed):
    rng = np.random.default_rng(seed)
    while True:                                   # a non-symmetric one, so Pi != Pi^T
        perm = rng.permutation(n)
        sign = rng.choice([-1.0, 1.0], n)
        p = np.zeros((n, n), np.float32)
        p[np.arange(n), perm] = sign
        if not np.array_equal(p, p.T):
            return p, perm, sign


@pytest.mark.parametrize("n", [2, 10, 64, 128])
def test_tq_fp64_rotation_on_a_signed_permutation(table, n):
    # with Pi a signed permutation every product is exact, so y = u Pi can be
    # written out by index: y[perm[i]] = sign[i] u[i]; a transposed Pi (u Pi^T)
    # or a dropped normalisation would not match
    p, perm, sign = _signed_permutation(n, n)
    rng = np.random.default_rng(7 + n)
    x = (rng.standard_normal((50, n)) * rng.lognormal(0, 1, (50, 1))).astype(np.float32)
    x[3] = 0.0
    cb = bgtq.scaled_codebook(table, 3, n)
    codes, nh, r, y = bgtq.tq_encode_fp64_rotation(x, p, cb)
    r64 = np.sqrt(np.sum(x.astype(np.float64) ** 2, -1))
    assert np.array_equal(r, r64.astype(np.float32))
    u = (x / np.where(r > 0, r, 1)[:, None].astype(np.float32)).astype(np.float32)
    want = np.zeros_like(u)
    want[:, perm] = u * sign[None, :].astype(np.float32)
    assert np.array_equal(y, want)
    assert np.array_equal(codes[r > 0], _brute_nearest(want, cb)[r > 0])
    assert codes[3].max() == 0 and float(nh[3]) == 0.0
    assert np.array_equal(nh, r.astype(np.float16))


def test_tq_fp64_rotation_agrees_with_the_fp32_chain(table):
    # the two encoders differ only in how y and r are rounded: a code may
    # differ only where y lies within a few fp32 ulps of a midpoint, and such
    # flips must be rare
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(21)
    flips = total = 0
    for n, b in ((8, 4), (30, 3), (128, 3), (64, 2)):
        x = (rng.standard_normal((600, n)) * rng.lognormal(0, 1, (600, 1))).astype(np.float32)
        cb = bgtq.scaled_codebook(table, b, n)
        c1, n1, r1, y1 = bgtq.tq_encode(x, pis[n], cb)
        c2, n2, r2, y2 = bgtq.tq_encode_fp64_rotation(x, pis[n], cb)
        assert np.max(np.abs(r1.astype(np.float64) / r2 - 1)) <= 4e-7
        assert np.max(np.abs(y1.astype(np.float64) - y2)) <= 1e-5
        diff = c1 != c2
        if diff.any():
            c64 = cb.astype(np.float64)
            mids = 0.5 * (c64[:-1] + c64[1:])
            lo = np.minimum(c1[diff], c2[diff])
            gap = np.abs(y2[diff].astype(np.float64) - mids[lo])
            ulp = np.spacing(np.abs(y2[diff])).astype(np.float64)
            assert np.all(gap <= 8 * ulp + np.abs(y1[diff].astype(np.float64) - y2[diff]))
            assert np.all(np.abs(c1[diff] - c2[diff]) == 1)
        flips += int(diff.sum())
        total += diff.size
        assert np.sum(n1 != n2) <= 0.01 * n1.size
    assert flips <= 1e-3 * total


# --------------------------------------------- dense dequantisation of a head

def test_dequantize_dense_equals_the_packed_cache_read_back(table):
    # dequantize_dense (no packing) against read_token of the cache that
    # append wrote (bit streams, norm slots, grouped layout): a gather or
    # scatter slip in either path breaks the equality
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(41)
    T, v_bits = 21, 3
    s = rng.lognormal(0, 2, 64)
    widths = bgtq.greedy_allocate(s, 1, 8, 192)
    sd = np.sqrt(np.concatenate([s, s]) / 2)
    k = (rng.standard_normal((T, 1, 128)) * sd).astype(np.float32)
    v = rng.standard_normal((T, 1, 128)).astype(np.float32)
    k[4] = 0.0
    cache = bgtq.new_cache(2, 1, 192, v_bits)
    slots = rng.permutation(32)[:T]
    bgtq.append(cache, k, v, slots, widths[None], v_bits, 192, pis, table)
    kh, vh = bgtq.dequantize_dense(k[:, 0], v[:, 0], widths, v_bits, pis, table)
    for t in range(T):
        page, sl = divmod(int(slots[t]), 16)
        kt, vt = bgtq.read_token(cache, page, sl, 0, widths, v_bits, 192, pis, table)
        # equal up to the summation order of the batched and single products
        assert np.max(np.abs(kh[t] - kt)) <= 1e-12 * max(1.0, np.max(np.abs(kt)))
        assert np.max(np.abs(vh[t] - vt)) <= 1e-12 * max(1.0, np.max(np.abs(vt)))
    assert np.all(kh[4] == 0)


def test_dequantize_dense_approaches_the_input_at_high_width(table):
    # at 8 bits per coordinate TQ-MSE keeps ~1e-4 of the energy as error;
    # a transposed rotation, a wrong dimension pairing or a dropped norm gives
    # errors of order one.  Both rotation paths are checked.
    pis = bgtq.tq_rotation_dict(*inputs.tq_rotations(128, "pin"))
    rng = np.random.default_rng(42)
    T = 40
    widths = np.concatenate([np.full(20, 8), np.full(44, 7)])
    rng.shuffle(widths)
    k = (rng.standard_normal((T, 128)) * rng.lognormal(0, 1, (T, 1))).astype(np.float32)
    v = (rng.standard_normal((T, 128)) * 3).astype(np.float32)
    for exact in (True, False):
        kh, vh = bgtq.dequantize_dense(k, v, widths, 8, pis, table, exact_chain=exact)
        ek = np.sum((kh - k) ** 2, -1) / np.sum(k.astype(np.float64) ** 2, -1)
        ev = np.sum((vh - v) ** 2, -1) / np.sum(v.astype(np.float64) ** 2, -1)
        assert ek.max() <= 20 * bgtq.C_TQ * 4.0 ** -7 and ev.max() <= 20 * bgtq.C_TQ * 4.0 ** -8
        assert ek.mean() <= bgtq.C_TQ * 4.0 ** -7


def test_value_codes_sit_in_slot_pairs():
    # the pair row of slots (2j, 2j+1) interleaves their codes channel by
    # channel; writing one slot keeps the partner's codes
    v_bits, total_bits = 3, 192
    lay = bgtq.tile_layout(total_bits, v_bits)
    tile = np.zeros(lay["tile"], np.uint8)
    rng = np.random.default_rng(11)
    even = rng.integers(0, 8, 128)
    odd = rng.integers(0, 8, 128)
    bgtq.write_v_codes(tile, 6, even, total_bits, v_bits)
    bgtq.write_v_codes(tile, 7, odd, total_bits, v_bits)
    o = lay["v_codes"] + 3 * 2 * lay["vb"]
    row = tile[o:o + 2 * lay["vb"]]
    # bit 6c + k of the row is bit k of slot 6's code of channel c (k < 3),
    # bit 6c + 3 + k that of slot 7
    bits = np.unpackbits(row, bitorder="little")
    for c in (0, 1, 5, 127):
        assert sum(int(bits[6 * c + k]) << k for k in range(3)) == even[c]
        assert sum(int(bits[6 * c + 3 + k]) << k for k in range(3)) == odd[c]
    # only that row is touched, and rewriting a slot leaves its partner alone
    assert not tile[:o].any() and not tile[o + 2 * lay["vb"]:].any()
    bgtq.write_v_codes(tile, 6, np.zeros(128, np.int64), total_bits, v_bits)
    assert np.array_equal(bgtq.read_v_codes(tile, 7, total_bits, v_bits), odd)
    assert not bgtq.read_v_codes(tile, 6, total_bits, v_bits).any()
