// Block-GTQ: grouped TQ-MSE key codes with per-RoPE-block widths, uniform
// TQ-MSE value codes, and fused decode attention over the packed cache.
//
// "RoPE-Aware Bit Allocation for KV-Cache Quantization":
//   prerequisites (TQ-MSE): normalise x, rotate by a shared orthogonal Pi,
//     scalar-quantise every rotated coordinate, keep the radius;
//   method step (3): RoPE blocks of equal width b form one sub-vector (the
//     blocks' post-RoPE coordinates concatenated) encoded at b bits/dim;
//   method step (4): values use uniform-width TQ-MSE;
//   Figure 2: persistent HBM holds packed code streams plus norms; the fused
//     kernel decodes only the current tile into kernel-local temporaries.
//
// Decode works in the TQ basis: <q_b, r c Pi^T> = r <q_b Pi, c>, so each
// query sub-vector is rotated once per CTA (q~_b = q_b Pi_n), a key
// contributes r_b * c[code] * q~ per coordinate, and values accumulate
// sum_s p_s r_s c[code] in the Pi_128 basis, rotated back once at the end.
#include <mutex>

#include "merge.cuh"

namespace kvq {

// Per-head layout of the grouped key sub-vectors (built from the widths).
struct BgtqLayout {
    int16_t dim[D];      // gathered position -> original dimension
    int16_t start[9];    // first position of the width-b group
    int16_t n[9];        // length of the width-b group (2 * blocks)
    int16_t bitstart[9]; // first code bit of the width-b group
    int total_bits;      // sum over positions of the widths
    int ok;              // widths all in 1..8
};

// Thread 0 fills the layout: groups in ascending width, blocks ascending
// inside a group, each block as (dim i, dim i + 64).
__device__ void build_layout(const int8_t* __restrict__ w, BgtqLayout& L) {
    int pos = 0, bit = 0, ok = 1;
    for (int i = 0; i < D / 2; ++i) ok &= (w[i] >= 1 && w[i] <= 8);
    for (int b = 1; b <= 8; ++b) {
        L.start[b] = (int16_t)pos;
        L.bitstart[b] = (int16_t)bit;
        for (int i = 0; i < D / 2; ++i)
            if (w[i] == b) {
                L.dim[pos++] = (int16_t)i;
                L.dim[pos++] = (int16_t)(i + D / 2);
            }
        L.n[b] = (int16_t)(pos - L.start[b]);
        bit += b * L.n[b];
    }
    L.total_bits = bit;
    L.ok = ok && pos == D;
}

__host__ __device__ inline int bgtq_kb(int total_bits) { return 4 * ((2 * total_bits + 31) / 32); }

// Scaled codebook fp32(C_b[c] / sqrt(n)), computed in fp64 then rounded once.
__device__ __forceinline__ float scaled_centroid(const double* __restrict__ cb, int b, int c, int n) {
    return __double2float_rn(cb[(b - 1) * 256 + c] / sqrt((double)n));
}

// Number of midpoints (c_k + c_{k+1}) / 2 (exact in fp64) strictly below y:
// the nearest centroid, ties to the lower index.
__device__ __forceinline__ int nearest_code(float y, const float* __restrict__ c, int levels) {
    int lo = 0, hi = levels - 1;
    const double yd = (double)y;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const double m = 0.5 * ((double)c[mid] + (double)c[mid + 1]);
        if (m < yd) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Group of gathered position p (1..8).
__device__ __forceinline__ int group_of(const BgtqLayout& L, int p) {
    int b = 1;
    while (b < 8 && !(p >= L.start[b] && p < L.start[b] + L.n[b])) ++b;
    return b;
}

// ------------------------------------------------------------------ append

struct AppendSmem {
    BgtqLayout L;
    float cb_k[8][256];
    float cb_v[256];
    float x[2][D];       // [0] gathered key, [1] value
    float u[2][D];       // normalised
    uint32_t words[2][32];
    uint16_t knorm[8];
    uint16_t vnorm;
};

__global__ void __launch_bounds__(256)
bgtq_append_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, int n_tok, int H_kv,
                   const int32_t* __restrict__ slot_mapping, const int8_t* __restrict__ widths, int total_bits,
                   int v_bits, const float* __restrict__ pi_table, const int64_t* __restrict__ pi_offsets,
                   const double* __restrict__ codebooks, uint8_t* __restrict__ cache, int64_t num_pages,
                   int32_t* __restrict__ err_count, int tok_per_cta, int tile_bytes) {
    __shared__ AppendSmem sm;
    const int h = blockIdx.y, tid = threadIdx.x;
    const int side = tid >> 7, p = tid & (D - 1);  // side 0: key position p, side 1: value channel p
    if (tid == 0) build_layout(widths + h * (D / 2), sm.L);
    __syncthreads();
    if (!sm.L.ok || sm.L.total_bits > 2 * total_bits) {
        if (tid == 0 && blockIdx.x == 0 && err_count) atomicAdd(err_count, 1);
        return;
    }
    for (int idx = tid; idx < 8 * 256; idx += 256) {
        const int b = idx / 256 + 1, c = idx % 256;
        if (c < (1 << b) && sm.L.n[b] > 0) sm.cb_k[b - 1][c] = scaled_centroid(codebooks, b, c, sm.L.n[b]);
    }
    for (int c = tid; c < (1 << v_bits); c += 256) sm.cb_v[c] = scaled_centroid(codebooks, v_bits, c, D);

    // this thread's coordinate: group width, start, length, index, code bit
    int b, st, n, j, bit;
    if (side == 0) {
        b = group_of(sm.L, p);
        st = sm.L.start[b];
        n = sm.L.n[b];
        j = p - st;
        bit = sm.L.bitstart[b] + j * b;
    } else {
        b = v_bits;
        st = 0;
        n = D;
        j = p;
        bit = p * v_bits;
    }
    const float* pi = pi_table + __ldg(pi_offsets + n);
    const int kb = bgtq_kb(total_bits), vb = 16 * v_bits;
    const int off_kn = PAGE * kb, off_vc = off_kn + PAGE * 16, off_vn = off_vc + PAGE * vb;
    const int64_t n_slots = num_pages * PAGE;
    const int t0 = blockIdx.x * tok_per_cta, t1 = min(n_tok, t0 + tok_per_cta);
    __syncthreads();

    for (int t = t0; t < t1; ++t) {
        const int slot = __ldg(slot_mapping + t);
        if (slot == -1) continue;
        if (slot < -1 || (int64_t)slot >= n_slots) {
            if (tid == 0 && h == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        const __nv_bfloat16* src = (side ? v : k) + ((size_t)t * H_kv + h) * D;
        sm.x[side][p] = __bfloat162float(src[side ? p : sm.L.dim[p]]);
        if (tid < 64) sm.words[tid >> 5][tid & 31] = 0u;
        if (tid < 8) sm.knorm[tid] = 0;
        __syncthreads();

        // r = sqrt(fp32 fma chain of squares), u = x / r
        const float* xs = sm.x[side] + st;
        float ss = 0.f;
        for (int i = 0; i < n; ++i) ss = __fmaf_rn(xs[i], xs[i], ss);
        const float r = __fsqrt_rn(ss);
        sm.u[side][p] = r > 0.f ? __fdiv_rn(sm.x[side][p], r) : 0.f;
        __syncthreads();

        // y_j = u Pi_n column j (fp32 fma chain), nearest scaled centroid
        const float* us = sm.u[side] + st;
        float y = 0.f;
#pragma unroll 16
        for (int i = 0; i < n; ++i) y = __fmaf_rn(us[i], __ldg(pi + (size_t)i * n + j), y);
        const uint32_t code = r > 0.f ? (uint32_t)nearest_code(y, side ? sm.cb_v : sm.cb_k[b - 1], 1 << b) : 0u;
        const int w = bit >> 5, sh = bit & 31;
        atomicOr(&sm.words[side][w], code << sh);
        if (sh + b > 32) atomicOr(&sm.words[side][w + 1], code >> (32 - sh));
        if (j == 0) {
            const uint16_t nh = __half_as_ushort(f16_sat(r));
            if (side) sm.vnorm = nh; else sm.knorm[b - 1] = nh;
        }
        __syncthreads();

        const int page = slot / PAGE, s = slot % PAGE;
        uint8_t* tile = cache + ((size_t)page * H_kv + h) * tile_bytes;
        if (tid < kb / 4) reinterpret_cast<uint32_t*>(tile + s * kb)[tid] = sm.words[0][tid];
        if (tid >= 64 && tid < 64 + vb / 4)
            reinterpret_cast<uint32_t*>(tile + off_vc + s * vb)[tid - 64] = sm.words[1][tid - 64];
        if (tid >= 128 && tid < 136) reinterpret_cast<uint16_t*>(tile + off_kn + 16 * s)[tid - 128] = sm.knorm[tid - 128];
        if (tid == 136) reinterpret_cast<uint16_t*>(tile + off_vn)[s] = sm.vnorm;
        __syncthreads();
    }
}

// ------------------------------------------------------------------ decode

constexpr int BG_WARPS = 4;
constexpr int BG_STAGES = 4;

struct BgDecodeSmem {
    BgtqLayout L;
    float cb_k[8][256];
    float cb_v[256];
    float q[8][D];          // q~ in gathered key order, times scale * log2(e)
    float qin[8][D];
    MergeSmem<BG_WARPS, 8> ms;
    uint64_t bar[BG_WARPS][BG_STAGES];
    float o_part[BG_WARPS][8][D];
};

__global__ void __launch_bounds__(128)
bgtq_decode_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int G, const uint8_t* __restrict__ cache,
                   int64_t num_pages, const int32_t* __restrict__ block_table, int max_pages,
                   const int32_t* __restrict__ context_lens, const int8_t* __restrict__ widths, int total_bits,
                   int v_bits, const float* __restrict__ pi_table, const int64_t* __restrict__ pi_offsets,
                   const double* __restrict__ codebooks, float scale_log2, float* __restrict__ out,
                   uint8_t* __restrict__ ws, int tile_bytes) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BgDecodeSmem& sm = *reinterpret_cast<BgDecodeSmem*>(smem_raw);
    uint8_t* ring = smem_raw + align_up(sizeof(BgDecodeSmem), 128);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, S = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* err_word = reinterpret_cast<uint32_t*>(ws);

    int ctx = __ldg(context_lens + b);
    ctx = max(0, min(ctx, max_pages * PAGE));
    const int n_pages = (ctx + PAGE - 1) / PAGE;
    const int pps = (n_pages + S - 1) / S;
    const int p_begin = min(split * pps, n_pages), p_end = min(p_begin + pps, n_pages);
    const int my_count = p_end - p_begin > warp ? (p_end - p_begin - warp + BG_WARPS - 1) / BG_WARPS : 0;
    const int32_t* bt = block_table + (size_t)b * max_pages;
    uint8_t* my_ring = ring + (size_t)warp * BG_STAGES * tile_bytes;

    if (lane == 0) {
        for (int s = 0; s < BG_STAGES; ++s) mbar_init(&sm.bar[warp][s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    auto issue = [&](int i) {  // lane 0 only
        const int p = p_begin + warp + BG_WARPS * i;
        const int pid = __ldg(bt + p);
        uint64_t* bar = &sm.bar[warp][i % BG_STAGES];
        if (pid < 0 || (int64_t)pid >= num_pages) {
            atomicOr(err_word, ERR_BAD_PAGE);
            mbar_arrive(bar);
        } else {
            mbar_arrive_expect_tx(bar, tile_bytes);
            bulk_g2s(my_ring + (size_t)(i % BG_STAGES) * tile_bytes, cache + ((size_t)pid * H_kv + h) * tile_bytes,
                     tile_bytes, bar);
        }
    };
    if (lane == 0)
        for (int i = 0; i < min(BG_STAGES, my_count); ++i) issue(i);

    // ---- per-head layout, codebooks and rotated queries
    if (tid == 0) build_layout(widths + h * (D / 2), sm.L);
    const __nv_bfloat16* qb = q + ((size_t)b * H_q + (size_t)h * G) * D;
    for (int idx = tid; idx < G * D; idx += 128) sm.qin[idx / D][idx % D] = __bfloat162float(qb[idx]);
    __syncthreads();
    const bool layout_ok = sm.L.ok && sm.L.total_bits <= 2 * total_bits;
    if (!layout_ok && tid == 0) atomicOr(err_word, ERR_BAD_WIDTHS);
    for (int idx = tid; idx < 8 * 256; idx += 128) {
        const int bb = idx / 256 + 1, c = idx % 256;
        if (c < (1 << bb) && sm.L.n[bb] > 0) sm.cb_k[bb - 1][c] = scaled_centroid(codebooks, bb, c, sm.L.n[bb]);
    }
    for (int c = tid; c < (1 << v_bits); c += 128) sm.cb_v[c] = scaled_centroid(codebooks, v_bits, c, D);
    if (layout_ok) {
        // q~ at gathered position p = tid: sum_i q[dim(st + i)] Pi_n[i][p - st]
        const int p = tid;
        const int bb = group_of(sm.L, p);
        const int st = sm.L.start[bb], n = sm.L.n[bb], j = p - st;
        const float* pi = pi_table + __ldg(pi_offsets + n);
        float acc[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
#pragma unroll 16
        for (int i = 0; i < n; ++i) {
            const float pv = __ldg(pi + (size_t)i * n + j);
            const int dm = sm.L.dim[st + i];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                if (jj < G) acc[jj] = fmaf(sm.qin[jj][dm], pv, acc[jj]);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (jj < G) sm.q[jj][p] = acc[jj] * scale_log2;
    }
    __syncthreads();

    const int kb = bgtq_kb(total_bits), vb = 16 * v_bits;
    const int off_kn = PAGE * kb, off_vc = off_kn + PAGE * 16, off_vn = off_vc + PAGE * vb;
    const int s_tok = lane & 15, half = lane >> 4;
    const uint32_t vmask = (1u << v_bits) - 1u;

    float mrun[8], lsum[8], oacc[8][4];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
        mrun[jj] = -CUDART_INF_F;
        lsum[jj] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[jj][e] = 0.f;
    }
    bool timed_out = false;

    for (int i = 0; i < my_count; ++i) {
        const int stage = i % BG_STAGES;
        const uint32_t parity = (i / BG_STAGES) & 1;
        if (!timed_out) {
            const bool okw = mbar_wait_bounded(&sm.bar[warp][stage], parity, WAIT_LIMIT_CYCLES);
            if (__any_sync(0xffffffffu, !okw)) {
                timed_out = true;
                if (lane == 0) atomicOr(err_word, ERR_TIMEOUT);
            }
        }
        if (timed_out) break;
        const uint8_t* tile = my_ring + (size_t)stage * tile_bytes;
        const int pg = p_begin + warp + BG_WARPS * i;
        const int pid = __ldg(bt + pg);
        const bool valid = layout_ok && pid >= 0 && (int64_t)pid < num_pages;
        const int n_tok = valid ? min(PAGE, ctx - pg * PAGE) : 0;

        // ---- QK: lane = (token s_tok, gathered positions of parity `half`)
        float dot[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) dot[jj] = 0.f;
        if (valid) {
            const uint8_t* rec = tile + s_tok * kb;
            const __half* kn = reinterpret_cast<const __half*>(tile + off_kn + 16 * s_tok);
            for (int bb = 1; bb <= 8; ++bb) {
                const int n = sm.L.n[bb];
                if (n == 0) continue;
                const float rb = __half2float(kn[bb - 1]);
                const int st = sm.L.start[bb], bs = sm.L.bitstart[bb];
                const uint32_t mask = (1u << bb) - 1u;
                const float* cb = sm.cb_k[bb - 1];
                for (int e = half; e < n; e += 2) {
                    const int bit = bs + e * bb;
                    const uint32_t lo = lds32(rec + 4 * (bit >> 5)), hi = lds32(rec + 4 * (bit >> 5) + 4);
                    const uint32_t code = __funnelshift_r(lo, hi, bit & 31) & mask;
                    const float val = rb * cb[code];
                    const int p = st + e;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        if (jj < G) dot[jj] = fmaf(val, sm.q[jj][p], dot[jj]);
                }
            }
        }
        // ---- online softmax over the page's 16 tokens (lanes s and s + 16 agree)
        float pr[8], corr[8];
        bool need = false;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            pr[jj] = 0.f;
            corr[jj] = 1.f;
            if (jj >= G) continue;
            float lg = dot[jj] + __shfl_xor_sync(0xffffffffu, dot[jj], 16);
            lg = s_tok < n_tok ? lg : -CUDART_INF_F;
            float pm = lg;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
            if (pm > mrun[jj]) {
                corr[jj] = exp2f(mrun[jj] - pm);
                mrun[jj] = pm;
                need = true;
            }
            const float mref = mrun[jj] == -CUDART_INF_F ? 0.f : mrun[jj];
            pr[jj] = exp2f(lg - mref);
            float ps = half == 0 ? pr[jj] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            lsum[jj] = fmaf(lsum[jj], corr[jj], ps);
        }
        if (need) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[jj][e] *= corr[jj];
        }
        // ---- PV: lane owns channels 4*lane .. 4*lane+3 (4*v_bits contiguous bits)
        const int vbit = 4 * lane * v_bits;
        for (int s = 0; s < n_tok; ++s) {
            const uint8_t* vrec = tile + off_vc + s * vb;
            const uint32_t lo = lds32(vrec + 4 * (vbit >> 5));
            const uint32_t hi = (vbit >> 5) + 1 < vb / 4 ? lds32(vrec + 4 * (vbit >> 5) + 4) : 0u;
            const uint32_t codes = __funnelshift_r(lo, hi, vbit & 31);
            const float rv = __half2float(reinterpret_cast<const __half*>(tile + off_vn)[s]);
            float cv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) cv[e] = sm.cb_v[(codes >> (e * v_bits)) & vmask];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (jj >= G) continue;
                const float wgt = __shfl_sync(0xffffffffu, pr[jj], s) * rv;
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[jj][e] = fmaf(wgt, cv[e], oacc[jj][e]);
            }
        }
        __syncwarp();
        if (lane == 0 && i + BG_STAGES < my_count) {
            fence_proxy_async_smem();
            issue(i + BG_STAGES);
        }
    }
    if (timed_out && lane == 0)
        for (int s = 0; s < BG_STAGES; ++s) (void)mbar_wait_bounded(&sm.bar[warp][s], 0, 1000000LL);

#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
        if (jj < G) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sm.o_part[warp][jj][4 * lane + e] = oacc[jj][e];
            if (lane == 0) {
                sm.ms.m_part[warp][jj] = mrun[jj];
                sm.ms.l_part[warp][jj] = lsum[jj];
            }
        }
    __syncthreads();
    finish_decode<BG_WARPS, 8>(sm.ms, sm.o_part, G, H_q, H_kv, gridDim.z, b, h, split, S, ws,
                               pi_table + __ldg(pi_offsets + D), out);
}

// ------------------------------------------------------------- calibration

// Method step (1): s_{h,i} = 1/2 E_{t,g in G(h)} ||q_{t,g}(i)||^2 +
// 1/2 E_t ||k_{t,h}(i)||^2 over a calibration prefix, block i = dims
// (i, i + d/2); and the paired estimate s*_{h,i} = E_{t,g} ||q(i)|| ||k(i)||
// (AM-GM keeps it at or below s).  CTA (h, chunk) takes tokens
// chunk * CAL_TOK .. + CAL_TOK: thread (i, lane4) every 4th of them.
// Products of bf16 values are exact in fp64 and the sums are fp64 (the
// paired term takes fp32 square roots); the 4 token lanes combine in a fixed
// order, and each CTA adds its share (already divided by the token counts)
// into the outputs with fp64 atomics.
constexpr int CAL_TOK = 256;

__global__ void __launch_bounds__(256)
bgtq_energy_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int T, int H_q, int H_kv,
                   double* __restrict__ scores, double* __restrict__ paired) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int L = D / 2;
    const int h = blockIdx.x, chunk = blockIdx.y;
    const int i = threadIdx.x % L, lane4 = threadIdx.x / L;
    const int G = H_q / H_kv;
    const int t0 = chunk * CAL_TOK, t1 = min(T, t0 + CAL_TOK);
    double qs = 0.0, ks = 0.0, ps = 0.0;
    for (int t = t0 + lane4; t < t1; t += 4) {
        const __nv_bfloat16* kr = k + ((size_t)t * H_kv + h) * D;
        const double ka = __bfloat162float(kr[i]), kb = __bfloat162float(kr[i + L]);
        const double kn = fma(ka, ka, kb * kb);  // bf16 products are exact in fp64
        ks += kn;
        const float kroot = sqrtf((float)kn);
        for (int g = 0; g < G; ++g) {
            const __nv_bfloat16* qr = q + ((size_t)t * H_q + (size_t)h * G + g) * D;
            const double qa = __bfloat162float(qr[i]), qb = __bfloat162float(qr[i + L]);
            const double qn = fma(qa, qa, qb * qb);
            qs += qn;
            ps += (double)(sqrtf((float)qn) * kroot);
        }
    }
    __shared__ double red[3][4][L];
    red[0][lane4][i] = qs;
    red[1][lane4][i] = ks;
    red[2][lane4][i] = ps;
    __syncthreads();
    if (lane4 == 0) {
        double a = 0.0, b = 0.0, c = 0.0;
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            a += red[0][l][i];
            b += red[1][l][i];
            c += red[2][l][i];
        }
        const double n_q = (double)T * G, n_k = (double)T;
        atomicAdd(scores + (size_t)h * L + i, 0.5 * a / n_q + 0.5 * b / n_k);
        if (paired) atomicAdd(paired + (size_t)h * L + i, c / n_q);
    }
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status bgtq_energy_scores(const void* q, const void* k, int T, int H_q, int H_kv, int d,
                                         double* scores, double* paired, void* stream) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_energy_scores: d=%d (only 128)", d);
    if (T < 0 || H_kv <= 0 || H_q <= 0 || H_q % H_kv || H_kv > 65535)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_energy_scores: T=%d H_q=%d H_kv=%d", T, H_q, H_kv);
    if (!scores || (T > 0 && (!q || !k)))
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_energy_scores: null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)H_kv * (D / 2) * sizeof(double);
    kvq_status s = kvq_check_cuda(cudaMemsetAsync(scores, 0, bytes, st), "bgtq_energy_scores: clearing scores");
    if (s != KVQ_OK) return s;
    if (paired) {
        s = kvq_check_cuda(cudaMemsetAsync(paired, 0, bytes, st), "bgtq_energy_scores: clearing paired");
        if (s != KVQ_OK) return s;
    }
    if (T == 0) return KVQ_OK;
    const int chunks = (T + CAL_TOK - 1) / CAL_TOK;
    if (chunks > 65535) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_energy_scores: T=%d too long", T);
    return kvq_check_cuda(launch_pdl(bgtq_energy_kernel, dim3(H_kv, chunks), dim3(256), 0, st,
                                     static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), T,
                                     H_q, H_kv, scores, paired),
                          "bgtq_energy_scores launch");
}

static kvq_status check_bgtq_common(const char* fn, int d, int H_kv, int total_bits, int v_bits,
                                    const float* pi_table) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: d=%d (only 128)", fn, d);
    if (H_kv <= 0 || H_kv > 65535) return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: H_kv=%d", fn, H_kv);
    if (bgtq_tile_bytes(total_bits, v_bits) == 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: total_bits=%d (64..512) v_bits=%d (1..8)", fn, total_bits,
                             v_bits);
    if (reinterpret_cast<uintptr_t>(pi_table) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: pi_table needs 16-byte alignment", fn);
    return KVQ_OK;
}

extern "C" kvq_status bgtq_append(const void* k, const void* v, int n_tok, int H_kv, int d, const int32_t* slot_mapping,
                                  const int8_t* widths, int total_bits, int v_bits, const float* pi_table,
                                  const int64_t* pi_offsets, const double* codebooks, void* cache, int64_t num_pages,
                                  int32_t* err_count, void* stream) {
    kvq_status st = check_bgtq_common("bgtq_append", d, H_kv, total_bits, v_bits, pi_table);
    if (st != KVQ_OK) return st;
    if (n_tok < 0 || num_pages <= 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_append: n_tok=%d num_pages=%lld", n_tok, (long long)num_pages);
    if (n_tok == 0) return KVQ_OK;
    if (!k || !v || !slot_mapping || !widths || !pi_table || !pi_offsets || !codebooks || !cache)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_append: null pointer");
    if (reinterpret_cast<uintptr_t>(cache) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_append: cache needs 16-byte alignment");
    const int tile = (int)bgtq_tile_bytes(total_bits, v_bits);
    int chunks = (152 * 4 + H_kv - 1) / H_kv;
    int per = (n_tok + chunks - 1) / chunks;
    per = per < 1 ? 1 : (per > 64 ? 64 : per);
    dim3 grid((n_tok + per - 1) / per, H_kv);
    bgtq_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), n_tok, H_kv, slot_mapping, widths,
        total_bits, v_bits, pi_table, pi_offsets, codebooks, static_cast<uint8_t*>(cache), num_pages, err_count, per,
        tile);
    return kvq_check_cuda(cudaGetLastError(), "bgtq_append launch");
}

extern "C" kvq_status bgtq_decode_attn(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                       int64_t num_pages, const int32_t* block_table, int max_pages_per_seq,
                                       const int32_t* context_lens, const int8_t* widths, int total_bits, int v_bits,
                                       const float* pi_table, const int64_t* pi_offsets, const double* codebooks,
                                       float scale, float* out, void* workspace, size_t workspace_bytes,
                                       int num_splits, void* stream) {
    kvq_status st = check_bgtq_common("bgtq_decode_attn", d, H_kv, total_bits, v_bits, pi_table);
    if (st != KVQ_OK) return st;
    if (B <= 0 || B > 65535 || H_q <= 0 || H_q % H_kv || max_pages_per_seq <= 0 || num_pages <= 0 || num_splits < 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: B=%d H_q=%d H_kv=%d max_pages=%d", B, H_q, H_kv,
                             max_pages_per_seq);
    const int G = H_q / H_kv;
    if (G > 8) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: GQA group %d > 8", G);
    if (!q || !cache || !block_table || !context_lens || !widths || !pi_table || !pi_offsets || !codebooks || !out ||
        !workspace)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: null pointer");
    if (reinterpret_cast<uintptr_t>(cache) % 16 || reinterpret_cast<uintptr_t>(workspace) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: cache and workspace need 16-byte alignment");
    const int S = num_splits > 0 ? num_splits : bgtq_decode_auto_splits(B, H_kv, max_pages_per_seq);
    if (S > MAX_SPLITS)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: num_splits=%d above %d", S, MAX_SPLITS);
    const size_t need = kvq_decode_workspace_bytes(B, H_q, H_kv, max_pages_per_seq, S);
    if (workspace_bytes < need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "bgtq_decode_attn: workspace %zu < %zu bytes", workspace_bytes, need);
    const int tile = (int)bgtq_tile_bytes(total_bits, v_bits);
    const size_t smem = align_up(sizeof(BgDecodeSmem), 128) + (size_t)BG_WARPS * BG_STAGES * tile;
    {
        // opt in once per device, to the largest tile any width budget gives
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        kvq_status s2 = kvq_check_cuda(cudaGetDevice(&dev), "bgtq_decode_attn: cudaGetDevice");
        if (s2 != KVQ_OK) return s2;
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !done[dev]) {
            const size_t max_smem =
                align_up(sizeof(BgDecodeSmem), 128) + (size_t)BG_WARPS * BG_STAGES * bgtq_tile_bytes(512, 8);
            s2 = kvq_check_cuda(
                cudaFuncSetAttribute(bgtq_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem),
                "bgtq_decode_attn smem attribute");
            if (s2 != KVQ_OK) return s2;
            if (dev >= 0 && dev < 64) done[dev] = true;
        }
    }
    dim3 grid(S, H_kv, B);
    bgtq_decode_kernel<<<grid, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(q), H_q, H_kv, G, static_cast<const uint8_t*>(cache), num_pages, block_table,
        max_pages_per_seq, context_lens, widths, total_bits, v_bits, pi_table, pi_offsets, codebooks,
        scale * 1.4426950408889634f, out, static_cast<uint8_t*>(workspace), tile);
    return kvq_check_cuda(cudaGetLastError(), "bgtq_decode_attn launch");
}
