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
