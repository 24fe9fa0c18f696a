// Block-GTQ: quantise-on-append (grouped TQ-MSE key codes with per-RoPE-block
// widths, uniform TQ-MSE value codes) and the calibration energy scores; the
// fused decode is in bgtq_decode.cu.
//
// "RoPE-Aware Bit Allocation for KV-Cache Quantization":
//   prerequisites (TQ-MSE): normalise x, rotate by a shared orthogonal Pi,
//     scalar-quantise every rotated coordinate, keep the radius;
//   method step (3): RoPE blocks of equal width b form one sub-vector (the
//     blocks' post-RoPE coordinates concatenated) encoded at b bits/dim;
//   method step (4): values use uniform-width TQ-MSE;
//   Figure 2: persistent HBM holds packed code streams plus norms.

#include "bgtq_common.cuh"

namespace kvq {

// ------------------------------------------------------------------ append

struct AppendSmem {
    BgtqLayout L;
    float cb_k[8][256];
    float cb_v[256];
    float x[2][D];       // [0] gathered key, [1] value
    float u[2][D];       // normalised
    uint32_t kw[32];     // the slot's key code stream
    uint32_t vw[64];     // the slot's value codes in their pair row (the partner's bits zero)
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
        bit = 2 * p * v_bits;  // within the slot pair's row; the odd slot's code follows the even one's
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
        if (tid < 32) sm.kw[tid] = 0u;
        if (tid >= 64 && tid < 128) sm.vw[tid - 64] = 0u;
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
        const int cbit = bit + (side ? (slot & 1) * v_bits : 0);
        const int w = cbit >> 5, sh = cbit & 31;
        uint32_t* words = side ? sm.vw : sm.kw;
        atomicOr(&words[w], code << sh);
        if (sh + b > 32) atomicOr(&words[w + 1], code >> (32 - sh));
        if (j == 0) {
            const uint16_t nh = __half_as_ushort(f16_sat(r));
            if (side) sm.vnorm = nh; else sm.knorm[b - 1] = nh;
        }
        __syncthreads();

        const int page = slot / PAGE, s = slot % PAGE;
        uint8_t* tile = cache + ((size_t)page * H_kv + h) * tile_bytes;
        if (tid < kb / 4) reinterpret_cast<uint32_t*>(tile + s * kb)[tid] = sm.kw[tid];
        if (tid >= 64 && tid < 64 + 2 * vb / 4) {
            // the pair row is shared with the partner slot, which this or
            // another CTA may write at the same time: clear and set only
            // this slot's bits, atomically
            const int wi = tid - 64;
            uint32_t mine = 0u;
            for (int q = 0; q < 32; ++q)
                if (((32 * wi + q) % (2 * v_bits)) / v_bits == (s & 1)) mine |= 1u << q;
            uint32_t* dst = reinterpret_cast<uint32_t*>(tile + off_vc + (s >> 1) * 2 * vb) + wi;
            atomicAnd(dst, ~mine);
            atomicOr(dst, sm.vw[wi] & mine);
        }
        if (tid >= 128 && tid < 136) reinterpret_cast<uint16_t*>(tile + off_kn + 16 * s)[tid - 128] = sm.knorm[tid - 128];
        if (tid == 136) reinterpret_cast<uint16_t*>(tile + off_vn)[s] = sm.vnorm;
        __syncthreads();
    }
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

kvq_status bgtq_check_common(const char* fn, int d, int H_kv, int total_bits, int v_bits, const float* pi_table) {
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
    kvq_status st = bgtq_check_common("bgtq_append", d, H_kv, total_bits, v_bits, pi_table);
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
