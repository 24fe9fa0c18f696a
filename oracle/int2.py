"""Rotated INT2 KV-cache quantisation and packed-cache decode (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows "Output-Aware Rotation for INT2 KV-Cache Quantization":
  §1 (introduction): INT2 stores 1/8 of BF16; all values of a quantisation
      group share one scale; the key is centred before rotation and
      quantisation, which shifts every logit of a query by the same constant
      and leaves the softmax unchanged.
  §3.1 Eq. (4): D_{R,c}(z) = Q2(zR; c, G) R^T, with R orthogonal, clip ratio
      c and group size G.  Readings used here: c scales the group's range
      ends (c = 1, the plain min/max range, by default), G = 32 consecutive
      rotated channels of one token, asymmetric levels min + code*scale,
      scale = (max - min)/3, both stored as fp16.
  §3 Eqs. (1)-(2): decode attention; the cache is consumed in the rotated
      basis: <q, k~> = <qR_k, Q2(z)> and o = (sum_s p_s Q2(w_s)) R_v^T.

Cache format (one 1536-byte tile per (page, KV head); pages of 16 slots):
  [   0,  512) K codes  16 slots x 32 B
  [ 512,  768) K meta   16 slots x 4 groups x (scale fp16, min fp16)
  [ 768, 1280) V codes  16 slots x 32 B
  [1280, 1408) V scales 8 slot pairs x 4 groups x (fp16 of slot 2j, of slot 2j+1)
  [1408, 1536) V mins   the same for the mins
  cache[page][kv_head] tiles, row-major.  Code record of a 128-channel
  rotated vector: byte 4*b + g (b = 0..7, g = 0..3) holds channels
  32*g + 4*b + c (c = 0..3) in bits 2c..2c+1.  The value meta is stored
  pair-major (a 4-byte word holds one group's scales, or mins, of two
  adjacent slots): a layout choice of this library, not of the method.
"""
from __future__ import annotations

import numpy as np

from . import attention
from .fp import chain_matvec_f32, f16_rn_sat

PAGE = 16
D = 128
GROUP = 32
N_GROUPS = D // GROUP
TILE_BYTES = 1536
OFF_K_CODES, OFF_K_META, OFF_V_CODES, OFF_V_META = 0, 512, 768, 1280
CODE_BYTES = 32
META_BYTES = 16


# --------------------------------------------------------------------------
# quantiser Q2 (one group of 32 rotated values)
# --------------------------------------------------------------------------

def quant_params(x32: np.ndarray, clip: float = 1.0):
    """fp16 (scale, min) of each group along the last axis (length 32).

    Clip ratio c (§3.1, Q2(.; c, G)): the group's range ends are scaled,
    min_c = c*min and max_c = c*max (fp32 products), so for c < 1 values
    beyond the clipped range saturate at the end codes; c = 1 is the plain
    min/max range.  Taken in the kernel's precision: the products, max - min
    and the division by 3 are fp32 operations rounded to nearest, then
    rounded to fp16 (saturating).
    """
    x32 = np.asarray(x32, dtype=np.float32)
    c = np.float32(clip)
    mn = (c * x32.min(axis=-1)).astype(np.float32)
    mx = (c * x32.max(axis=-1)).astype(np.float32)
    rng = (mx - mn).astype(np.float32)
    s = (rng / np.float32(3.0)).astype(np.float32)
    return f16_rn_sat(s), f16_rn_sat(mn)


def quant_codes(x32: np.ndarray, scale_h: np.ndarray, min_h: np.ndarray) -> np.ndarray:
    """Nearest of the four levels min + c*scale (c = 0..3), ties to the lower
    code: the code counts the thresholds min + (c + 1/2)*scale, c = 0, 1, 2,
    that lie strictly below x (exact in fp64).  scale == 0 gives code 0."""
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    sc = np.asarray(scale_h, dtype=np.float16).astype(np.float64)[..., None]
    mn = np.asarray(min_h, dtype=np.float16).astype(np.float64)[..., None]
    code = np.zeros(x.shape, dtype=np.uint8)
    for c in range(3):
        code += (mn + (c + 0.5) * sc < x).astype(np.uint8)
    return np.where(sc == 0.0, 0, code).astype(np.uint8)


def quantize(z32: np.ndarray, clip: float = 1.0):
    """Q2 of rotated vectors [..., 128] -> (codes [...,128] u8,
    scale [...,4] f16, min [...,4] f16), clip ratio `clip`."""
    z32 = np.asarray(z32, dtype=np.float32)
    g = z32.reshape(z32.shape[:-1] + (N_GROUPS, GROUP))
    scale_h, min_h = quant_params(g, clip)
    codes = quant_codes(g, scale_h, min_h)
    return codes.reshape(z32.shape), scale_h, min_h


def dequantize_f32(codes: np.ndarray, scale_h: np.ndarray, min_h: np.ndarray) -> np.ndarray:
    """min + code*scale as one fp32 fused multiply-add (exact product, one
    rounding of the sum), [..., 128] fp32: the value a reader of the cache
    gets in fp32."""
    c = np.asarray(codes, dtype=np.float64)
    c = c.reshape(c.shape[:-1] + (N_GROUPS, GROUP))
    out = (np.asarray(min_h, np.float16).astype(np.float64)[..., None]
           + c * np.asarray(scale_h, np.float16).astype(np.float64)[..., None])   # exact in fp64
    return out.astype(np.float32).reshape(out.shape[:-2] + (D,))


def dequantize(codes: np.ndarray, scale_h: np.ndarray, min_h: np.ndarray) -> np.ndarray:
    """min + code*scale in fp64, [..., 128]."""
    c = np.asarray(codes, dtype=np.float64)
    c = c.reshape(c.shape[:-1] + (N_GROUPS, GROUP))
    out = (np.asarray(min_h, np.float16).astype(np.float64)[..., None]
           + c * np.asarray(scale_h, np.float16).astype(np.float64)[..., None])
    return out.reshape(out.shape[:-2] + (D,))


# --------------------------------------------------------------------------
# record packing
# --------------------------------------------------------------------------

def pack_codes(codes: np.ndarray) -> np.ndarray:
    """codes [..., 128] in 0..3 -> bytes [..., 32] (group-interleaved)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape[:-1] + (CODE_BYTES,), dtype=np.uint8)
    for b in range(8):
        for g in range(N_GROUPS):
            v = np.zeros(c.shape[:-1], dtype=np.uint8)
            for cc in range(4):
                v |= (c[..., 32 * g + 4 * b + cc] & 3) << (2 * cc)
            out[..., 4 * b + g] = v
    return out


def unpack_codes(rec: np.ndarray) -> np.ndarray:
    rec = np.asarray(rec, dtype=np.uint8)
    out = np.zeros(rec.shape[:-1] + (D,), dtype=np.uint8)
    for b in range(8):
        for g in range(N_GROUPS):
            byte = rec[..., 4 * b + g]
            for cc in range(4):
                out[..., 32 * g + 4 * b + cc] = (byte >> (2 * cc)) & 3
    return out


def pack_meta(scale_h: np.ndarray, min_h: np.ndarray) -> np.ndarray:
    """[..., 4] fp16 pairs -> [..., 16] bytes: (scale, min) per group,
    little-endian."""
    pair = np.stack([np.asarray(scale_h, np.float16), np.asarray(min_h, np.float16)], axis=-1)
    return pair.reshape(pair.shape[:-2] + (8,)).view(np.uint8)


def unpack_meta(raw: np.ndarray):
    h = np.ascontiguousarray(raw, dtype=np.uint8).view(np.float16)
    h = h.reshape(h.shape[:-1] + (N_GROUPS, 2))
    return h[..., 0], h[..., 1]


def meta_bytes(side: int, s: int) -> np.ndarray:
    """Tile byte offsets of slot s's 16-byte meta record (pack_meta order:
    per group scale lo, hi, min lo, hi) for side 0 (keys) or 1 (values)."""
    if side == 0:
        return OFF_K_META + META_BYTES * s + np.arange(META_BYTES)
    pair, half = divmod(s, 2)
    idx = []
    for g in range(N_GROUPS):
        base = OFF_V_META + 16 * pair + 4 * g + 2 * half
        idx += [base, base + 1, base + 128, base + 129]
    return np.asarray(idx)


# --------------------------------------------------------------------------
# quantise-on-append
# --------------------------------------------------------------------------

def rotate_keys(k: np.ndarray, mu32: np.ndarray, r32: np.ndarray, exact_chain=True):
    """Centred, rotated keys z = (k - mu) R (row-vector convention, Eq. 4).

    k: [n, d] (bf16 values), mu32: [d] fp32, r32: [d, d] fp32.
    Returns (z32 used for the codes, z64 in fp64).  With exact_chain the fp32
    value reproduces the kernels' fma chain bit for bit; otherwise it is the
    fp64 product rounded to fp32 (large sampled checks).
    """
    kc32 = (np.asarray(k, np.float32) - np.asarray(mu32, np.float32)).astype(np.float32)
    z64 = kc32.astype(np.float64) @ np.asarray(r32, np.float32).astype(np.float64)
    z32 = chain_matvec_f32(kc32, r32) if exact_chain else z64.astype(np.float32)
    return z32, z64


def rotate_values(v: np.ndarray, r32: np.ndarray, exact_chain=True):
    v32 = np.asarray(v, np.float32)
    w64 = v32.astype(np.float64) @ np.asarray(r32, np.float32).astype(np.float64)
    w32 = chain_matvec_f32(v32, r32) if exact_chain else w64.astype(np.float32)
    return w32, w64


def new_cache(num_pages: int, h_kv: int) -> np.ndarray:
    return np.zeros((num_pages, h_kv, TILE_BYTES), dtype=np.uint8)


def append(cache, k, v, slot_mapping, mu32, rk32, rv32, exact_chain=True, clip=1.0):
    """Quantise-on-append into the paged cache (in place).

    k, v: [n, H_kv, d] (bf16 values); slot_mapping[n] = page*16 + slot,
    -1 skips the token; mu32 [H_kv, d]; rk32, rv32 [H_kv, d, d] fp32;
    clip: the clip ratio c of Q2 (keys and values alike).
    Returns dict with the fp32 rotated vectors z, w ([n, H_kv, d]).
    """
    k = np.asarray(k)
    v = np.asarray(v)
    n, h_kv, d = k.shape
    z_all = np.zeros((n, h_kv, d), np.float32)
    w_all = np.zeros((n, h_kv, d), np.float32)
    sm = np.asarray(slot_mapping, dtype=np.int64)
    keep = sm >= 0
    for h in range(h_kv):
        z32, _ = rotate_keys(k[keep, h], mu32[h], rk32[h], exact_chain)
        w32, _ = rotate_values(v[keep, h], rv32[h], exact_chain)
        z_all[keep, h] = z32
        w_all[keep, h] = w32
        for side, src, off_c in ((0, z32, OFF_K_CODES), (1, w32, OFF_V_CODES)):
            codes, sc, mn = quantize(src, clip)
            recs = pack_codes(codes)
            metas = pack_meta(sc, mn)
            for i, slot in enumerate(sm[keep]):
                page, s = divmod(int(slot), PAGE)
                cache[page, h, off_c + CODE_BYTES * s: off_c + CODE_BYTES * (s + 1)] = recs[i]
                cache[page, h, meta_bytes(side, s)] = metas[i]
    return {"z": z_all, "w": w_all}


def read_tokens(cache, page_ids, n_tokens, h):
    """Dequantised rotated (K^, V^) of the first n_tokens of a page list for
    KV head h, fp64 [n_tokens, d] each."""
    if n_tokens == 0:
        return np.zeros((0, D)), np.zeros((0, D))
    n_pages = (n_tokens + PAGE - 1) // PAGE
    tiles = cache[np.asarray(page_ids[:n_pages], dtype=np.int64), h]      # [P, 1536]

    def side(which, off_c):
        recs = tiles[:, off_c: off_c + PAGE * CODE_BYTES].reshape(-1, CODE_BYTES)
        meta = tiles[:, np.stack([meta_bytes(which, s) for s in range(PAGE)])].reshape(-1, META_BYTES)
        sc, mn = unpack_meta(meta)
        return dequantize(unpack_codes(recs), sc, mn)[:n_tokens]

    return side(0, OFF_K_CODES), side(1, OFF_V_CODES)


# --------------------------------------------------------------------------
# packed-cache decode attention
# --------------------------------------------------------------------------

def decode(q, cache, block_table, ctx_lens, mu32, rk32, rv32, scale, h_kv, window=None):
    """Decode attention over the packed INT2 cache, fp64, as the plain
    definition: the effective cached key and value of Eq. (4),
        k~_s = Q2((k_s - mu) R_k) R_k^T + mu,   v~_s = Q2(v_s R_v) R_v^T,
    then Eqs. (1)-(2) over s < ctx_lens[b] with logit scale `scale`.

    window: None, or (k_win, v_win, win_lens) with k_win, v_win
    [B, W, H_kv, d] (bf16 values) and win_lens[B] <= W.  The INT2 paper keeps
    a small window of tokens in BF16 (§3.1; the Block-GTQ page keeps 4 sink
    and 128 recent tokens, Table 6).  Window tokens are attended exactly, in
    the original basis, together with the cached tokens: the softmax runs
    over the union of the s < ctx_lens[b] cached tokens and the first
    win_lens[b] window tokens.  A window token is not also in the INT2
    range; which tokens go where is the caller's choice.

    q: [B, H_q, d] (bf16 values); mu32 [H_kv, d]; rk32, rv32 [H_kv, d, d].
    Returns [B, H_q, d].  (Adding mu back shifts every logit of a query by
    the same constant, so the softmax does not depend on it.)
    """
    q = np.asarray(q, dtype=np.float64)
    B, h_q, d = q.shape
    rk = np.asarray(rk32, np.float32).astype(np.float64)
    rv = np.asarray(rv32, np.float32).astype(np.float64)
    mu = np.asarray(mu32, np.float32).astype(np.float64)
    sc = float(np.float32(scale))
    out = np.zeros((B, h_q, d))
    for b in range(B):
        T = int(ctx_lens[b])
        kt = np.zeros((T, h_kv, d))
        vt = np.zeros((T, h_kv, d))
        for h in range(h_kv):
            kz, vw = read_tokens(cache, block_table[b], T, h)
            kt[:, h] = kz @ rk[h].T + mu[h]
            vt[:, h] = vw @ rv[h].T
        if window is not None:
            k_win, v_win, win_lens = window
            wl = int(win_lens[b])
            kt = np.concatenate([kt, np.asarray(k_win[b, :wl], np.float64)], axis=0)
            vt = np.concatenate([vt, np.asarray(v_win[b, :wl], np.float64)], axis=0)
        out[b] = attention.gqa_decode(q[b], kt, vt, sc)
    return out


def storage_bytes_per_token_head() -> dict:
    """Byte accounting of one cached token for one KV head."""
    return {"k_codes": CODE_BYTES, "k_meta": META_BYTES,
            "v_codes": CODE_BYTES, "v_meta": META_BYTES,
            "total": 2 * (CODE_BYTES + META_BYTES), "bf16_kv": 2 * D * 2}
