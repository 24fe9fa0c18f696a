"""Block-GTQ: RoPE-block bit allocation with TQ-MSE codes (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows "RoPE-Aware Bit Allocation for KV-Cache Quantization":
  prerequisites, TQ-MSE: normalise a non-zero x, apply a shared orthogonal
      rotation, scalar-quantise every rotated coordinate, keep the radius;
      E||x - x^||^2 <= ||x||^2 C_TQ 4^-b.  The page renders C_TQ as
      sqrt(3*pi/2) = 2.171; read here as sqrt(3)*pi/2 = 2.721, the
      Panter-Dite high-rate constant of a Gaussian source, which Lloyd-Max
      quantisers approach from below (with 2.171 the law fails for b >= 4).
  prerequisites, greedy allocation / Theorem 1: start every block at b_min,
      repeatedly give one more bit to the block with the largest marginal
      gain Delta_i(b_i) = s_i 4^-b_i - s_i 4^-(b_i+1) = (3/4) s_i 4^-b_i, until
      the budget is spent or b_max is reached; optimal for
      J(b) = sum_i s_i 4^-b_i over integer widths.
  method steps (3)-(4): blocks with equal width form G_b = {i : b_i = b};
      their post-RoPE key blocks are concatenated and TQ-MSE-encoded at b
      bits per dimension; values use uniform-width TQ-MSE.
  core method: the RoPE logit is a sum over 2-D blocks and the key-error
      logit bound is |K(q,k) - K(q,k^)| <= sum_i ||q(i)|| ||e_k(i)||.
  method step (1): label-free block energy scores from a calibration
      prefix, s_i = 1/2 E||q(i)||^2 + 1/2 E||k(i)||^2 (energy_scores).

Readings (the pages leave these open): block i is the rotate-half pair of
dims (i, i + d/2); x_b lists the blocks of G_b in ascending order, each as
(x[i], x[i+d/2]); the scalar quantiser is the Lloyd-Max codebook of N(0,1)
at b bits scaled by 1/sqrt(n) for an n-dim sub-vector (rotated unit-vector
coordinates have variance 1/n); nearest centroid with ties to the lower
index; norm kept as fp16; Pi_n is one Haar orthogonal matrix per length n.

Cache format (one tile per (page, KV head), 16 slots; KB = k code bytes,
VB = 16 * v_bits):
  [0, 16*KB)             K codes, dense LSB-first bit stream per slot:
                         groups by ascending width b = 1..8, coordinates in
                         order, b bits each, value LSB first
  [16*KB, +16*16)        K norms: 8 fp16 per slot, entry b-1 = width-b group
                         (0 when the group is empty)
  [.., +16*VB)           V codes by slot pair: pair j = slots (2j, 2j+1)
                         holds 2*VB bytes, an LSB-first stream of 128
                         entries in channel order, each the slot-2j code
                         then the slot-2j+1 code (v_bits bits each)
  [.., +16*2)            V norm fp16 per slot
KB = 4 * ceil(2 * total_bits / 32) with total_bits the per-head width budget.
The pages fix what is stored (code streams plus norms), not the byte order;
the value codes of two slots sit side by side so that a reader can take
one channel of two tokens as one 2*v_bits-bit field.
"""
from __future__ import annotations

import functools

import numpy as np
from scipy.special import ndtr, ndtri

from . import attention
from .fp import chain_matvec_f32, chain_sumsq_f32, f16_rn_sat

D = 128
L_BLOCKS = D // 2
PAGE = 16
B_MAX_WIDTH = 8
C_TQ = np.sqrt(3.0) * np.pi / 2.0


# --------------------------------------------------------------------------
# Gaussian Lloyd-Max codebooks
# --------------------------------------------------------------------------

def _cell_mass(a, b):
    """P(a < X < b) for X ~ N(0,1), computed on the side of the small tail."""
    return np.where(a >= 0, ndtr(-a) - ndtr(-b),
                    np.where(b <= 0, ndtr(b) - ndtr(a), 1.0 - ndtr(a) - ndtr(-b)))


def _pdf(x):
    xx = np.where(np.isinf(x), 0.0, x)
    return np.where(np.isinf(x), 0.0, np.exp(-0.5 * xx * xx) / np.sqrt(2.0 * np.pi))


@functools.lru_cache(maxsize=None)
def lloyd_max_gaussian(b: int) -> np.ndarray:
    """Centroids (ascending, fp64) of the 2^b-level Lloyd-Max quantiser of
    N(0,1), by plain Lloyd iteration: thresholds at the midpoints of adjacent
    centroids, centroids at the conditional means E[X | cell].  Starts at the
    quantile midpoints; stops when no centroid moves by more than 1e-14 or
    when the movement has stopped shrinking (fp64 noise floor)."""
    n = 2 ** b
    c = ndtri((np.arange(n) + 0.5) / n)
    best, since = np.inf, 0
    for _ in range(1_000_000):
        t = 0.5 * (c[:-1] + c[1:])
        lo = np.concatenate([[-np.inf], t])
        hi = np.concatenate([t, [np.inf]])
        cn = (_pdf(lo) - _pdf(hi)) / _cell_mass(lo, hi)
        move = float(np.max(np.abs(cn - c)))
        c = cn
        if move < 1e-14:
            break
        if move < 0.5 * best:
            best, since = move, 0
        else:
            since += 1
            if since > 20000 and best < 1e-12:
                break
    return c


def lloyd_max_table() -> np.ndarray:
    """[8, 256] fp64: row b-1 holds the 2^b centroids of width b, rest 0."""
    t = np.zeros((B_MAX_WIDTH, 256))
    for b in range(1, B_MAX_WIDTH + 1):
        t[b - 1, : 2 ** b] = lloyd_max_gaussian(b)
    return t


def scaled_codebook(table: np.ndarray, b: int, n: int) -> np.ndarray:
    """fp32 centroids for an n-dim sub-vector at width b: round_f32(C_b / sqrt(n))
    (fp64 division, one rounding to fp32)."""
    return (table[b - 1, : 2 ** b] / np.sqrt(np.float64(n))).astype(np.float32)


def nearest_codes(y32: np.ndarray, cb32: np.ndarray) -> np.ndarray:
    """Index of the nearest centroid, ties to the lower index: the number of
    midpoints (c_k + c_{k+1})/2 (exact in fp64) strictly below y."""
    y = np.asarray(y32, np.float32).astype(np.float64)
    c = np.asarray(cb32, np.float32).astype(np.float64)
    mids = 0.5 * (c[:-1] + c[1:])
    return (y[..., None] > mids).sum(axis=-1).astype(np.int64)


# --------------------------------------------------------------------------
# greedy RoPE-block allocator
# --------------------------------------------------------------------------

def energy_scores(q, k, h_kv: int):
    """Block energy scores of a calibration prefix (method step (1)):
        s_{h,i} = 1/2 E_{t, g in G(h)} ||q_{t,g}(i)||^2 + 1/2 E_t ||k_{t,h}(i)||^2,
    block i = dims (i, i + d/2), G(h) the query heads reading KV head h; and
    the paired estimate
        s*_{h,i} = E_{t, g in G(h)} ||q_{t,g}(i)|| ||k_{t,h}(i)||,
    which AM-GM (||q|| ||k|| <= (||q||^2 + ||k||^2) / 2, token by token)
    keeps at or below s (technical novelty (2): s* <= s).

    q: [T, H_q, d], k: [T, H_kv, d] (bf16 values); returns (s, s_star), each
    [H_kv, d/2] fp64.  T = 0 gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    T, h_q, d = q.shape
    L = d // 2
    g = h_q // h_kv
    if T == 0:
        return np.zeros((h_kv, L)), np.zeros((h_kv, L))
    qn = (q[..., :L] ** 2 + q[..., L:] ** 2).reshape(T, h_kv, g, L)   # ||q_{t,g}(i)||^2
    kn = k[..., :L] ** 2 + k[..., L:] ** 2                               # ||k_{t,h}(i)||^2
    s = 0.5 * qn.mean(axis=(0, 2)) + 0.5 * kn.mean(axis=0)
    s_star = (np.sqrt(qn) * np.sqrt(kn)[:, :, None, :]).mean(axis=(0, 2))
    return s, s_star


def greedy_allocate(scores, b_min: int, b_max: int, total_bits: int) -> np.ndarray:
    """Integer widths b_i in [b_min, b_max] with sum <= total_bits.

    Each step gives one bit to the block with the largest marginal gain
    (3/4) s_i 4^-b_i; the common factor 3/4 does not change the arg-max, so
    s_i 4^-b_i (an exact power-of-two scaling in fp64) is compared.  Ties go
    to the lowest block index.  Stops when the budget is spent or every block
    is at b_max.
    """
    s = np.asarray(scores, dtype=np.float64)
    b = np.full(s.shape[0], b_min, dtype=np.int64)
    budget = int(total_bits) - b_min * s.shape[0]
    while budget > 0:
        gain = np.where(b < b_max, np.ldexp(s, -2 * b), -np.inf)
        i = int(np.argmax(gain))
        if not np.isfinite(gain[i]):
            break
        b[i] += 1
        budget -= 1
    return b


def objective(scores, widths) -> float:
    """J(b) = sum_i s_i 4^-b_i."""
    return float(np.sum(np.asarray(scores, np.float64) * 4.0 ** (-np.asarray(widths, np.float64))))


# --------------------------------------------------------------------------
# grouping and TQ-MSE
# --------------------------------------------------------------------------

def width_groups(widths):
    """[(b, blocks ascending)] for every width b = 1..8 (empty lists kept)."""
    w = np.asarray(widths)
    return [(b, [int(i) for i in np.nonzero(w == b)[0]]) for b in range(1, B_MAX_WIDTH + 1)]


def gather(x: np.ndarray, blocks) -> np.ndarray:
    """Concatenate RoPE blocks: (x[i0], x[i0+64], x[i1], x[i1+64], ...)."""
    idx = []
    for i in blocks:
        idx += [i, i + L_BLOCKS]
    return np.asarray(x)[..., idx]


def scatter(xb: np.ndarray, blocks, out: np.ndarray):
    for j, i in enumerate(blocks):
        out[..., i] = xb[..., 2 * j]
        out[..., i + L_BLOCKS] = xb[..., 2 * j + 1]


def tq_encode(x32: np.ndarray, pi32: np.ndarray, cb32: np.ndarray):
    """TQ-MSE of sub-vectors x [..., n] fp32 in the kernel's precision:
    r = sqrt(fp32 fma-chain sum of squares), u = x / r (fp32), y = u Pi (fp32
    fma chain), code = nearest scaled centroid, norm = fp16(r).  r == 0 gives
    codes 0 and norm 0.  Returns (codes, norm_f16, r32, y32)."""
    x32 = np.asarray(x32, np.float32)
    r = np.sqrt(chain_sumsq_f32(x32)).astype(np.float32)
    safe = np.where(r > 0, r, np.float32(1.0)).astype(np.float32)
    u = (x32 / safe[..., None]).astype(np.float32)
    y = chain_matvec_f32(u, pi32)
    codes = nearest_codes(y, cb32)
    codes = np.where((r > 0)[..., None], codes, 0)
    return codes, f16_rn_sat(r), r, y


def tq_encode_fp64_rotation(x32: np.ndarray, pi32: np.ndarray, cb32: np.ndarray):
    """TQ-MSE with the norm and rotation taken in fp64 and rounded to fp32
    before the code decision (for long contexts, where the fp32 chain
    emulation is too slow; rare ties may then differ from the kernels)."""
    x32 = np.asarray(x32, np.float32)
    r = np.sqrt(np.sum(x32.astype(np.float64) ** 2, axis=-1)).astype(np.float32)
    safe = np.where(r > 0, r, np.float32(1.0)).astype(np.float32)
    u = (x32 / safe[..., None]).astype(np.float32)
    y = (u.astype(np.float64) @ np.asarray(pi32, np.float32).astype(np.float64)).astype(np.float32)
    codes = np.where((r > 0)[..., None], nearest_codes(y, cb32), 0)
    return codes, f16_rn_sat(r), r, y


def dequantize_dense(k32, v32, widths, v_bits, pis, table, exact_chain=True):
    """Dequantised keys and values [T, d] (fp64, original basis) of one KV
    head, without packing: grouped TQ-MSE keys (method step 3) and uniform
    TQ-MSE values (step 4)."""
    enc = tq_encode if exact_chain else tq_encode_fp64_rotation
    k32 = np.asarray(k32, np.float32)
    kh = np.zeros(k32.shape, np.float64)
    for b, bl in width_groups(widths):
        if not bl:
            continue
        n = 2 * len(bl)
        cb = scaled_codebook(table, b, n)
        codes, nh, _, _ = enc(gather(k32, bl), pis[n], cb)
        scatter(tq_decode(codes, nh, pis[n], cb), bl, kh)
    cbv = scaled_codebook(table, v_bits, D)
    codes, nh, _, _ = enc(np.asarray(v32, np.float32), pis[D], cbv)
    return kh, tq_decode(codes, nh, pis[D], cbv)


def tq_decode(codes, norm_f16, pi32, cb32) -> np.ndarray:
    """x^ = r * (c[codes] Pi^T), fp64."""
    c = np.asarray(cb32, np.float32).astype(np.float64)[np.asarray(codes)]
    pi = np.asarray(pi32, np.float32).astype(np.float64)
    return np.asarray(norm_f16, np.float16).astype(np.float64)[..., None] * (c @ pi.T)


# --------------------------------------------------------------------------
# bit streams and the paged format
# --------------------------------------------------------------------------

def pack_bits(values, widths, n_bytes: int) -> np.ndarray:
    """Dense LSB-first bit stream of unsigned values with per-value widths."""
    out = np.zeros(n_bytes, dtype=np.uint8)
    pos = 0
    for val, w in zip(values, widths):
        for k in range(int(w)):
            if (int(val) >> k) & 1:
                out[pos // 8] |= np.uint8(1 << (pos % 8))
            pos += 1
    assert pos <= 8 * n_bytes
    return out


def unpack_bits(stream, widths) -> np.ndarray:
    stream = np.asarray(stream, np.uint8)
    vals, pos = [], 0
    for w in widths:
        v = 0
        for k in range(int(w)):
            v |= ((int(stream[pos // 8]) >> (pos % 8)) & 1) << k
            pos += 1
        vals.append(v)
    return np.asarray(vals, dtype=np.int64)


def k_code_bytes(total_bits: int) -> int:
    return 4 * ((2 * int(total_bits) + 31) // 32)


def v_code_bytes(v_bits: int) -> int:
    return D * int(v_bits) // 8


def tile_layout(total_bits: int, v_bits: int) -> dict:
    kb, vb = k_code_bytes(total_bits), v_code_bytes(v_bits)
    off = {"k_codes": 0, "kb": kb, "vb": vb}
    off["k_norms"] = PAGE * kb
    off["v_codes"] = off["k_norms"] + PAGE * 16
    off["v_norms"] = off["v_codes"] + PAGE * vb
    off["tile"] = off["v_norms"] + PAGE * 2
    return off


def v_pair_offset(total_bits: int, v_bits: int, slot: int) -> int:
    """Byte offset, in a tile, of the value-code pair row holding `slot`."""
    lay = tile_layout(total_bits, v_bits)
    return lay["v_codes"] + (slot // 2) * 2 * lay["vb"]


def read_v_codes(tile, slot: int, total_bits: int, v_bits: int) -> np.ndarray:
    """The 128 value codes of one slot of a tile."""
    o = v_pair_offset(total_bits, v_bits, slot)
    pair = unpack_bits(tile[o:o + 2 * v_code_bytes(v_bits)], [v_bits] * (2 * D)).reshape(D, 2)
    return pair[:, slot % 2]


def write_v_codes(tile, slot: int, codes, total_bits: int, v_bits: int):
    """Store one slot's 128 value codes, keeping its pair partner's."""
    o = v_pair_offset(total_bits, v_bits, slot)
    n = 2 * v_code_bytes(v_bits)
    pair = unpack_bits(tile[o:o + n], [v_bits] * (2 * D)).reshape(D, 2)
    pair[:, slot % 2] = codes
    tile[o:o + n] = pack_bits(pair.reshape(-1), [v_bits] * (2 * D), n)


def new_cache(num_pages, h_kv, total_bits, v_bits):
    return np.zeros((num_pages, h_kv, tile_layout(total_bits, v_bits)["tile"]), np.uint8)


def encode_key(k32: np.ndarray, widths, pis: dict, table: np.ndarray):
    """Grouped TQ-MSE of one key [d] (fp32).  Returns (code list in stream
    order, width list, norms f16[8], y per group)."""
    vals, wl = [], []
    norms = np.zeros(B_MAX_WIDTH, np.float16)
    ys = {}
    for b, blocks in width_groups(widths):
        if not blocks:
            continue
        n = 2 * len(blocks)
        codes, nh, _, y = tq_encode(gather(k32, blocks), pis[n], scaled_codebook(table, b, n))
        vals += list(codes)
        wl += [b] * n
        norms[b - 1] = nh
        ys[b] = y
    return vals, wl, norms, ys


def append(cache, k, v, slot_mapping, widths, v_bits, total_bits, pis, table):
    """Quantise-on-append (in place).  k, v: [n, H_kv, d] bf16 values;
    widths [H_kv, 64]; pis {n: Pi_n fp32}; table [8, 256] fp64 codebooks."""
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    n, h_kv, _ = k.shape
    lay = tile_layout(total_bits, v_bits)
    kb = lay["kb"]
    cbv = scaled_codebook(table, v_bits, D)
    for t in range(n):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        page, s = divmod(slot, PAGE)
        for h in range(h_kv):
            vals, wl, norms, _ = encode_key(k[t, h], widths[h], pis, table)
            cache[page, h, s * kb:(s + 1) * kb] = pack_bits(vals, wl, kb)
            o = lay["k_norms"] + 16 * s
            cache[page, h, o:o + 16] = norms.view(np.uint8)
            codes, nh, _, _ = tq_encode(v[t, h], pis[D], cbv)
            write_v_codes(cache[page, h], s, codes, total_bits, v_bits)
            o = lay["v_norms"] + 2 * s
            cache[page, h, o:o + 2] = np.asarray([nh], np.float16).view(np.uint8)


def read_token(cache, page, slot, h, widths, v_bits, total_bits, pis, table):
    """Dequantised (k^, v^) [d] fp64 of one cached token, original basis."""
    lay = tile_layout(total_bits, v_bits)
    kb = lay["kb"]
    tile = cache[page, h]
    kh = np.zeros(D)
    groups = [(b, bl) for b, bl in width_groups(widths) if bl]
    stream = tile[slot * kb:(slot + 1) * kb]
    wl = []
    for b, bl in groups:
        wl += [b] * (2 * len(bl))
    vals = unpack_bits(stream, wl)
    norms = tile[lay["k_norms"] + 16 * slot: lay["k_norms"] + 16 * slot + 16].view(np.float16)
    pos = 0
    for b, bl in groups:
        n = 2 * len(bl)
        xb = tq_decode(vals[pos:pos + n], norms[b - 1], pis[n], scaled_codebook(table, b, n))
        scatter(xb, bl, kh)
        pos += n
    vcodes = read_v_codes(tile, slot, total_bits, v_bits)
    o = lay["v_norms"] + 2 * slot
    vn = tile[o:o + 2].view(np.float16)[0]
    vh = tq_decode(vcodes, vn, pis[D], scaled_codebook(table, v_bits, D))
    return kh, vh


def decode(q, cache, block_table, ctx_lens, widths, v_bits, total_bits, pis, table, scale, h_kv):
    """Decode attention over the packed Block-GTQ cache as the plain
    definition: dequantise every cached key and value to the original
    (post-RoPE) basis, then GQA attention (Eqs. 1-2 of the INT2 page's
    preliminaries) with logit scale `scale`.  Returns [B, H_q, d] fp64."""
    q = np.asarray(q, np.float64)
    B, h_q, d = q.shape
    out = np.zeros((B, h_q, d))
    for b in range(B):
        T = int(ctx_lens[b])
        kt = np.zeros((T, h_kv, d))
        vt = np.zeros((T, h_kv, d))
        for s in range(T):
            page = int(block_table[b][s // PAGE])
            for h in range(h_kv):
                kt[s, h], vt[s, h] = read_token(cache, page, s % PAGE, h, widths[h], v_bits,
                                                total_bits, pis, table)
        out[b] = attention.gqa_decode(q[b], kt, vt, float(np.float32(scale)))
    return out


def tq_rotation_dict(table_f64: np.ndarray, offsets: np.ndarray) -> dict:
    """{n: Pi_n fp32} from the flat table the input generator produces."""
    out = {}
    for n in range(2, len(offsets)):
        if offsets[n] >= 0:
            out[n] = table_f64[offsets[n]: offsets[n] + n * n].reshape(n, n).astype(np.float32)
    return out
