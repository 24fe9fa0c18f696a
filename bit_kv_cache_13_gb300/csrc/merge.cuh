// Pieces shared by the decode kernels: the query rotation prologue and the
// split-K finish.
//
// Split-K finish: each warp of a CTA leaves, per query head jj < G, its
// running maximum m (base-2 logits), normaliser l and unnormalised output o'
// (rotated basis) in shared memory.  finish_decode combines the warps,
// publishes the CTA's split partial (m, l, o') to the workspace, and the last
// CTA of the (sequence, KV head) to arrive -- decided by an atomic ticket,
// nobody waits -- merges the S split partials with the log-sum-exp rule
//     M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  O = sum_s o'_s 2^(m_s - M),
// rotates o = (O / L) Rot^T once (o_i = sum_j o'_j Rot[i][j]) and writes it.
// The ticket is reset to zero so the workspace is ready for the next call.
// Every global read in these paths is issued many-at-a-time (warps split
// the rows / splits, float4 loads) so their latency overlaps.
#pragma once

#include <math_constants.h>

#include "kvq_common.cuh"

namespace kvq {

constexpr int MAX_SPLITS = 256;

template <int NWARPS>
struct MergeSmem {
    float m_part[NWARPS][8];
    float l_part[NWARPS][8];
    float o_final[8][D];
    float red[NWARPS][8][D];    // cross-warp partial sums
    float fac[8][MAX_SPLITS];   // per-split weights 2^(m_s - M)
    float Mh[8], Lh[8];
    int is_last;
};

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// qr[jj][c] = sum_i qin[jj][i] * R[i][c] * factor for jj < G (128 threads).
// Warp w takes rows 32w .. 32w+31, lane takes columns 4*lane .. 4*lane+3.
template <int NWARPS>
__device__ __forceinline__ void rotate_rows(const float (*qin)[D], const float* __restrict__ R, int G, float factor,
                                            float (*qr)[D], MergeSmem<NWARPS>& ms) {
    static_assert(NWARPS * 32 == D, "one warp per 32 rows");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float4 acc[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
    for (int ii = 0; ii < 32; ++ii) {
        const int i = 32 * warp + ii;
        const float4 r = ldg4(R + (size_t)i * D + 4 * lane);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (jj < G) {
                const float x = qin[jj][i];
                acc[jj].x = fmaf(x, r.x, acc[jj].x);
                acc[jj].y = fmaf(x, r.y, acc[jj].y);
                acc[jj].z = fmaf(x, r.z, acc[jj].z);
                acc[jj].w = fmaf(x, r.w, acc[jj].w);
            }
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
        if (jj < G) *reinterpret_cast<float4*>(&ms.red[warp][jj][4 * lane]) = acc[jj];
    __syncthreads();
    const int c = threadIdx.x;
    for (int jj = 0; jj < G; ++jj) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) s += ms.red[w][jj][c];
        qr[jj][c] = s * factor;
    }
    __syncthreads();
}

// 128 threads; o_part[w][jj][c] is warp w's o'.  Rot is row-major [D][D]
// fp32, 16-byte aligned.  S <= MAX_SPLITS.
template <int NWARPS>
__device__ __forceinline__ void finish_decode(MergeSmem<NWARPS>& ms, const float (*o_part)[8][D], int G, int H_q,
                                              int H_kv, int B, int b, int h, int split, int S, uint8_t* ws,
                                              const float* __restrict__ Rot, float* __restrict__ out) {
    const int c = threadIdx.x, warp = c >> 5, lane = c & 31;
    int32_t* tickets = reinterpret_cast<int32_t*>(ws + WS_HEADER);
    float* partials = reinterpret_cast<float*>(ws + WS_HEADER + tickets_bytes(B, H_kv));
    const size_t head0 = (size_t)b * H_q + (size_t)h * G;

    // ---- warps -> this CTA's split partial
    for (int jj = 0; jj < G; ++jj) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, ms.m_part[w][jj]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < NWARPS; ++w) {
                const float f = exp2f(ms.m_part[w][jj] - M);
                L = fmaf(ms.l_part[w][jj], f, L);
                O = fmaf(o_part[w][jj][c], f, O);
            }
        }
        float* part = partials + ((head0 + jj) * S + split) * PART_STRIDE;
        part[4 + c] = O;
        if (c == 0) {
            part[0] = M;
            part[1] = L;
        }
    }
    __threadfence();
    __syncthreads();
    if (c == 0) {
        const int prev = atomicAdd(tickets + (size_t)b * H_kv + h, 1);
        ms.is_last = prev == S - 1;
    }
    __syncthreads();
    if (!ms.is_last) return;
    __threadfence();

    // ---- last CTA: split weights (one warp per head, lanes over splits)
    for (int jj = warp; jj < G; jj += NWARPS) {
        const float* base = partials + (head0 + jj) * S * PART_STRIDE;
        float M = -CUDART_INF_F;
        for (int s = lane; s < S; s += 32) {
            const float m = __ldcg(base + (size_t)s * PART_STRIDE);
            ms.fac[jj][s] = m;
            M = fmaxf(M, m);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int s = lane; s < S; s += 32) {
            const float f = M == -CUDART_INF_F ? 0.f : exp2f(ms.fac[jj][s] - M);
            ms.fac[jj][s] = f;
            L = fmaf(__ldcg(base + (size_t)s * PART_STRIDE + 1), f, L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            ms.Mh[jj] = M;
            ms.Lh[jj] = L;
        }
    }
    __syncthreads();
    // ---- weighted sum of the split outputs: warp w takes splits w, w+4, ...
    {
        float4 acc[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s = warp; s < S; s += NWARPS) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                if (jj < G) {
                    const float f = ms.fac[jj][s];
                    const float4 o = ldcg4(partials + ((head0 + jj) * S + s) * PART_STRIDE + 4 + 4 * lane);
                    acc[jj].x = fmaf(f, o.x, acc[jj].x);
                    acc[jj].y = fmaf(f, o.y, acc[jj].y);
                    acc[jj].z = fmaf(f, o.z, acc[jj].z);
                    acc[jj].w = fmaf(f, o.w, acc[jj].w);
                }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (jj < G) *reinterpret_cast<float4*>(&ms.red[warp][jj][4 * lane]) = acc[jj];
    }
    __syncthreads();
    for (int jj = 0; jj < G; ++jj) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) s += ms.red[w][jj][c];
        const float L = ms.Lh[jj];
        ms.o_final[jj][c] = L > 0.f ? s / L : 0.f;
    }
    __syncthreads();
    // ---- o_c = sum_j o'_j Rot[c][j]
    const float* row = Rot + (size_t)c * D;
    float acc[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
#pragma unroll
    for (int j4 = 0; j4 < D / 4; ++j4) {
        const float4 rv = ldg4(row + 4 * j4);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (jj < G) {
                const float* o = &ms.o_final[jj][4 * j4];
                acc[jj] = fmaf(o[0], rv.x, fmaf(o[1], rv.y, fmaf(o[2], rv.z, fmaf(o[3], rv.w, acc[jj]))));
            }
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
        if (jj < G) out[(head0 + jj) * D + c] = acc[jj];
    if (c == 0) tickets[(size_t)b * H_kv + h] = 0;
}

}  // namespace kvq
