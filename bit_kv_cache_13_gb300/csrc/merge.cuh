// Pieces shared by the decode kernels: the query rotation prologue and the
// split-K finish.
//
// Split-K finish: each warp of a CTA leaves, per query head jj < G, its
// running maximum m (base-2 logits), normaliser l and unnormalised output o'
// (rotated basis) in shared memory.  finish_decode combines the warps,
// publishes the CTA's split partial (m, l, o') to the workspace, and the last
// CTA of the (sequence, KV head) to arrive -- decided by an atomic ticket,
// nobody waits -- merges the S split partials with the log-sum-exp rule
//     M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  O = sum_s O_s 2^(m_s - M),
// and writes o = O / L.  The output rotation o = o' Rot^T is linear, so
// every CTA applies it to its own partial (O_s = o'_s Rot^T, o_i = sum_j
// o'_j Rot[i][j]) before publishing it: that work runs in parallel across
// the splits instead of in the one CTA that finishes last.
// The ticket is reset to zero so the workspace is ready for the next call.
// Every global read in these paths is issued many-at-a-time (warps split
// the rows / splits, float4 loads) so their latency overlaps.
//
// NW is the CTA's warp count.  A 128 x 128 rotation is shared by
// RotSplit<NW>::NR warps of RotSplit<NW>::RPW rows each: all four warps of a
// 4-warp CTA (32 rows each), eight warps of a larger one (16 rows each).
#pragma once

#include <math_constants.h>

#include "kvq_common.cuh"

namespace kvq {

constexpr int MAX_SPLITS = 256;

template <int NW>
struct RotSplit {
    static constexpr int NR = NW < 8 ? NW : 8;
    static constexpr int RPW = D / NR;
    static_assert(NR * RPW == D && (RPW == 16 || RPW == 32), "rotation split");
};

// Rows of R a rotating warp holds in registers at once: all of its rows,
// except 16 of 32 for head groups of 8 (register budget).
template <int NW, int MAXG>
struct RowPrefetch {
    static constexpr int N = (RotSplit<NW>::RPW == 32 && MAXG > 4) ? 16 : RotSplit<NW>::RPW;
};

// MAXG: the largest query-head group the kernel instance handles (G <= MAXG).
// 16-byte aligned: o_final and red are read and written as float4 rows.
template <int NW, int MAXG>
struct __align__(16) MergeSmem {
    float m_part[NW + 1][MAXG];  // per warp, and one more row for a lone token's partial
    float l_part[NW + 1][MAXG];
    float o_final[MAXG][D];
    float red[RotSplit<NW>::NR][MAXG][D];  // cross-warp partial sums
    float fac[MAXG][MAX_SPLITS];           // per-split maxima, then weights 2^(m_s - M)
    float lsp[MAXG][MAX_SPLITS];           // per-split normalisers
    float Mh[MAXG], Lh[MAXG];
    int is_last;
};

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// 2^x with the hardware approximation (relative error ~2^-22); -inf gives 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The first N rows of this warp's share of R (rows RPW*w .. RPW*w+N-1),
// columns 4*lane .. 4*lane+3, for the rotating warps w < NR: issued together
// so their latencies overlap (call early, use later).
template <int NW, int N>
__device__ __forceinline__ void load_rows(const float* __restrict__ R, float4 (&rr)[N]) {
    constexpr int NR = RotSplit<NW>::NR, RPW = RotSplit<NW>::RPW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= NR) return;
#pragma unroll
    for (int ii = 0; ii < N; ++ii) rr[ii] = ldg4(R + (size_t)(RPW * warp + ii) * D + 4 * lane);
}

// qr[jj][c] = sum_i qin[jj][i] * R[i][c] * factor for jj < G (all NW warps
// call it), with the first N of each rotating warp's rows of R already in rr
// (load_rows); the rest are loaded here.
template <int NW, int MAXG, int N>
__device__ __forceinline__ void rotate_rows(const float (*qin)[D], const float* __restrict__ R, const float4 (&rr)[N],
                                            int G, float factor, float (*qr)[D], MergeSmem<NW, MAXG>& ms) {
    constexpr int NR = RotSplit<NW>::NR, RPW = RotSplit<NW>::RPW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < NR) {
        float4 acc[MAXG];
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        auto accumulate = [&](int i, float4 r) {
#pragma unroll
            for (int jj = 0; jj < MAXG; ++jj)
                if (jj < G) {
                    const float x = qin[jj][i];
                    acc[jj].x = fmaf(x, r.x, acc[jj].x);
                    acc[jj].y = fmaf(x, r.y, acc[jj].y);
                    acc[jj].z = fmaf(x, r.z, acc[jj].z);
                    acc[jj].w = fmaf(x, r.w, acc[jj].w);
                }
        };
#pragma unroll
        for (int ii = 0; ii < N; ++ii) accumulate(RPW * warp + ii, rr[ii]);
        if constexpr (N < RPW) {
            float4 r2[RPW - N];
#pragma unroll
            for (int ii = 0; ii < RPW - N; ++ii) r2[ii] = ldg4(R + (size_t)(RPW * warp + N + ii) * D + 4 * lane);
#pragma unroll
            for (int ii = 0; ii < RPW - N; ++ii) accumulate(RPW * warp + N + ii, r2[ii]);
        }
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj)
            if (jj < G) *reinterpret_cast<float4*>(&ms.red[warp][jj][4 * lane]) = acc[jj];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int jj = idx / D, c = idx % D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NR; ++w) s += ms.red[w][jj][c];
        qr[jj][c] = s * factor;
    }
    __syncthreads();
}

// NW*32 threads; o_part[w][jj][c] is warp w's o'.  Rot is row-major [D][D]
// fp32, 16-byte aligned; with ROTATE false, o' is already in the output
// basis and Rot is not read.  S <= MAX_SPLITS, G <= MAXG.
template <int NW, int MAXG, bool ROTATE = true>
__device__ __forceinline__ void finish_decode(MergeSmem<NW, MAXG>& ms, const float (*o_part)[MAXG][D], int G, int H_q,
                                              int H_kv, int B, int b, int h, int split, int S, uint8_t* ws,
                                              const float* __restrict__ Rot, float* __restrict__ out) {
    constexpr int NR = RotSplit<NW>::NR, RPW = RotSplit<NW>::RPW, RP = RowPrefetch<NW, MAXG>::N;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t* tickets = reinterpret_cast<int32_t*>(ws + WS_HEADER);
    float* partials = reinterpret_cast<float*>(ws + WS_HEADER + tickets_bytes(B, H_kv));
    const size_t head0 = (size_t)b * H_q + (size_t)h * G;
    const size_t unit = (size_t)b * H_kv + h;

    // ---- warps -> this CTA's split partial (M, L, unnormalised o')
    // rows of Rot this warp rotates, columns 4*lane .. +3: coalesced, issued now
    float4 rr[RP];
    if constexpr (ROTATE) load_rows<NW, RP>(Rot, rr);
    // per (warp, head) weight 2^(m_w - M) in place of m_w, and the head's M, L
    if (tid < G) {
        const int jj = tid;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ms.m_part[w][jj]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = M == -CUDART_INF_F ? 0.f : ex2(ms.m_part[w][jj] - M);
            ms.m_part[w][jj] = f;
            L = fmaf(ms.l_part[w][jj], f, L);
        }
        ms.Mh[jj] = M;
        ms.Lh[jj] = L;
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int jj = idx / D, c = idx % D;
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) O = fmaf(o_part[w][jj][c], ms.m_part[w][jj], O);
        ms.o_final[jj][c] = O;
    }
    __syncthreads();
    // ---- rotate this partial: O_i = sum_j o'_j Rot[i][j] for the rows i of
    // this warp.  Each lane forms the partial dots of its 4 columns with RP
    // rows; a reduce-scatter over the lanes then leaves each row's full dot
    // in one lane (RP - 1 shuffles per head and RP rows, after a fold of the
    // two half-warps when RP = 16).  Heads go two at a time so their shuffle
    // chains overlap (the second of a pair past G is computed and dropped).
    if constexpr (!ROTATE) {
        // already in the output basis: publish o' as it is
        for (int idx = tid; idx < G * D; idx += NW * 32) {
            const int jj = idx / D, c = idx % D;
            float* part = partials + ((head0 + jj) * S + split) * PART_STRIDE;
            part[4 + c] = ms.o_final[jj][c];
            if (c == 0) {
                part[0] = ms.Mh[jj];
                part[1] = ms.Lh[jj];
            }
        }
    } else if (warp < NR) {
#pragma unroll
        for (int pass = 0; pass < RPW / RP; ++pass) {
            if (pass > 0) {
#pragma unroll
                for (int ii = 0; ii < RP; ++ii)
                    rr[ii] = ldg4(Rot + (size_t)(RPW * warp + RP * pass + ii) * D + 4 * lane);
            }
            for (int jj = 0; jj < G; jj += 2) {
                const int jb = jj + 1 < MAXG ? jj + 1 : jj;
                const float4 oa = *reinterpret_cast<const float4*>(&ms.o_final[jj][4 * lane]);
                const float4 ob = *reinterpret_cast<const float4*>(&ms.o_final[jb][4 * lane]);
                float va[RP], vb[RP];
#pragma unroll
                for (int ii = 0; ii < RP; ++ii) {
                    va[ii] = fmaf(oa.x, rr[ii].x, fmaf(oa.y, rr[ii].y, fmaf(oa.z, rr[ii].z, oa.w * rr[ii].w)));
                    vb[ii] = fmaf(ob.x, rr[ii].x, fmaf(ob.y, rr[ii].y, fmaf(ob.z, rr[ii].z, ob.w * rr[ii].w)));
                }
                if constexpr (RP == 16) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        va[k] += __shfl_xor_sync(0xffffffffu, va[k], 16);
                        vb[k] += __shfl_xor_sync(0xffffffffu, vb[k], 16);
                    }
                }
#pragma unroll
                for (int off = RP / 2; off >= 1; off >>= 1) {
                    const bool upper = lane & off;
#pragma unroll
                    for (int k = 0; k < off; ++k) {
                        const float sa = upper ? va[k] : va[k + off], ka = upper ? va[k + off] : va[k];
                        const float sb = upper ? vb[k] : vb[k + off], kb = upper ? vb[k + off] : vb[k];
                        va[k] = ka + __shfl_xor_sync(0xffffffffu, sa, off);
                        vb[k] = kb + __shfl_xor_sync(0xffffffffu, sb, off);
                    }
                }
                const int row = 4 + RPW * warp + RP * pass + (lane & (RP - 1));
                float* pa = partials + ((head0 + jj) * S + split) * PART_STRIDE;
                if (RP == 32 || lane < 16) pa[row] = va[0];
                if (tid == 0 && pass == 0) {
                    pa[0] = ms.Mh[jj];
                    pa[1] = ms.Lh[jj];
                }
                if (jj + 1 < G) {
                    float* pb = partials + ((head0 + jj + 1) * S + split) * PART_STRIDE;
                    if (RP == 32 || lane < 16) pb[row] = vb[0];
                    if (tid == 0 && pass == 0) {
                        pb[0] = ms.Mh[jj + 1];
                        pb[1] = ms.Lh[jj + 1];
                    }
                }
            }
        }
    }
    // publish: the barrier orders every thread's partial writes before
    // thread 0's release-acquire ticket; in the last CTA, the barrier after
    // the ticket orders all its reads of the other partials after it
    __syncthreads();
    if (tid == 0) ms.is_last = atomic_add_acq_rel_gpu(tickets + unit, 1) == S - 1;
    __syncthreads();
    if (!ms.is_last) return;

    // ---- last CTA: merge the S split partials of each head in one pass.
    // Warp jj takes head jj; the first run of split outputs is loaded
    // together with the (m, l) pairs, the weights 2^(m_s - M) pass through
    // shared memory, and each lane sums its 4 channels over the runs.
    constexpr int CH = NW >= 8 ? 32 : 16;  // split outputs in flight per lane
    for (int jj = warp; jj < G; jj += NW) {
        const float* ph = partials + (head0 + jj) * S * PART_STRIDE;
        float4 ov[CH];
        auto load_run = [&](int s0) {
#pragma unroll
            for (int k = 0; k < CH; ++k)
                ov[k] = s0 + k < S ? ldcg4(ph + (size_t)(s0 + k) * PART_STRIDE + 4 + 4 * lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        load_run(0);
        float M = -CUDART_INF_F;
        for (int s = lane; s < S; s += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(ph + (size_t)s * PART_STRIDE));
            ms.fac[jj][s] = ml.x;
            ms.lsp[jj][s] = ml.y;
            M = fmaxf(M, ml.x);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int s = lane; s < S; s += 32) {
            const float f = M == -CUDART_INF_F ? 0.f : ex2(ms.fac[jj][s] - M);
            ms.fac[jj][s] = f;
            L = fmaf(ms.lsp[jj][s], f, L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        __syncwarp();
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < S; s0 += CH) {
            if (s0 > 0) load_run(s0);
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const float f = s0 + k < S ? ms.fac[jj][s0 + k] : 0.f;
                acc.x = fmaf(f, ov[k].x, acc.x);
                acc.y = fmaf(f, ov[k].y, acc.y);
                acc.z = fmaf(f, ov[k].z, acc.z);
                acc.w = fmaf(f, ov[k].w, acc.w);
            }
        }
        float* o = out + (head0 + jj) * D + 4 * lane;
        o[0] = L > 0.f ? acc.x / L : 0.f;
        o[1] = L > 0.f ? acc.y / L : 0.f;
        o[2] = L > 0.f ? acc.z / L : 0.f;
        o[3] = L > 0.f ? acc.w / L : 0.f;
    }
    if (tid == 0) tickets[unit] = 0;
}


// ---------------------------------------------------------------------------
// Page-granular split-K (INT2 decode).  A CTA publishes one unrotated
// partial (m, l, o') per (sequence, KV head) unit it worked on; the last CTA
// of a unit merges them and applies the output rotation once.

// Combines the NW warps' (m, l, o') of this CTA: per head jj < G, Mh = max_w
// m_w, Lh = sum_w l_w 2^(m_w - Mh) and o_final = sum_w 2^(m_w - Mh) o_w.
// Every thread of the CTA calls it once the warps' (m, l, o') are in shared
// memory (after a barrier); each thread forms the weights of its own head,
// so one barrier, at the end, suffices.
// ROWS (NW or NW + 1) rows of (m, l, o') are combined.
template <int NW, int MAXG, int ROWS = NW>
__device__ __forceinline__ void merge_warps(MergeSmem<NW, MAXG>& ms, const float (*o_part)[MAXG][D], int G) {
    static_assert(ROWS <= NW + 1, "merge rows");
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int jj = idx / D, c = idx % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < ROWS; ++w) M = fmaxf(M, ms.m_part[w][jj]);
        float O = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < ROWS; ++w) {
            const float f = M == -CUDART_INF_F ? 0.f : ex2(ms.m_part[w][jj] - M);
            O = fmaf(o_part[w][jj][c], f, O);
            L = fmaf(ms.l_part[w][jj], f, L);
        }
        ms.o_final[jj][c] = O;
        if (c == 0) {
            ms.Mh[jj] = M;
            ms.Lh[jj] = L;
        }
    }
    __syncthreads();
}

// Writes G heads of (Mh, Lh, src) to a partial slot: head jj at
// slot + jj * PART_STRIDE as (m, l, -, -, o[128]).  With empty set, writes
// an empty partial (m = -inf, l = 0, o = 0) instead.
template <int NW, int MAXG>
__device__ __forceinline__ void publish_slot(const MergeSmem<NW, MAXG>& ms, const float (*src)[D], int G,
                                             float* __restrict__ slot, bool empty) {
    for (int idx = threadIdx.x; idx < G * (D / 4); idx += NW * 32) {
        const int jj = idx / (D / 4), c4 = idx % (D / 4);
        float4 v = empty ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(&src[jj][4 * c4]);
        *reinterpret_cast<float4*>(slot + (size_t)jj * PART_STRIDE + 4 + 4 * c4) = v;
        if (c4 == 0) {
            slot[(size_t)jj * PART_STRIDE] = empty ? -CUDART_INF_F : ms.Mh[jj];
            slot[(size_t)jj * PART_STRIDE + 1] = empty ? 0.f : ms.Lh[jj];
        }
    }
}

// Publishes under the unit's ticket: true in the one CTA that arrives last
// (of `expected`).  The barrier before orders every thread's partial writes
// before thread 0's release-acquire add; the barrier after orders the last
// CTA's reads of the other partials after it.
template <int NW, int MAXG>
__device__ __forceinline__ bool arrive_last(MergeSmem<NW, MAXG>& ms, int32_t* ticket, int expected) {
    __syncthreads();
    if (threadIdx.x == 0) ms.is_last = atomic_add_acq_rel_gpu(ticket, 1) == expected - 1;
    __syncthreads();
    return ms.is_last;
}

// Rotates this CTA's merged partial o_final (G heads) by Rot^T -- O_i =
// sum_j o'_j Rot[i][j], Rot row-major [D][D], 16-byte aligned -- and writes
// it, with (Mh, Lh), to a partial slot (head jj at slot + jj * PART_STRIDE as
// m, l, -, -, O[128]).  With direct set, the partial is the unit's only
// one, and slot is the heads' output rows [G][D]: out[jj][i] = O_i / Lh (0
// when Lh = 0) is written instead, the value the merge of that single
// partial gives (the merge path multiplies by exactly 1).  rr holds each rotating
// warp's first rows of Rot (load_rows, issued early so their latency is
// hidden).  Each lane forms the partial dots of its 4 columns with its warp's
// rows, and a reduce-scatter over the lanes leaves each row's full dot in
// one lane (heads two at a time so their shuffle chains overlap).  All
// threads call it.
template <int NW, int MAXG>
__device__ __forceinline__ void rotate_publish(const MergeSmem<NW, MAXG>& ms, float4 (&rr)[RowPrefetch<NW, MAXG>::N],
                                               int G, const float* __restrict__ Rot, float* __restrict__ slot,
                                               bool direct = false) {
    const int stride = direct ? D : PART_STRIDE, first = direct ? 0 : 4;
    constexpr int NR = RotSplit<NW>::NR, RPW = RotSplit<NW>::RPW, RP = RowPrefetch<NW, MAXG>::N;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < NR) {
#pragma unroll
        for (int pass = 0; pass < RPW / RP; ++pass) {
            if (pass > 0) {
#pragma unroll
                for (int ii = 0; ii < RP; ++ii)
                    rr[ii] = ldg4(Rot + (size_t)(RPW * warp + RP * pass + ii) * D + 4 * lane);
            }
            for (int jj = 0; jj < G; jj += 2) {
                const int jb = jj + 1 < MAXG ? jj + 1 : jj;
                const float4 oa = *reinterpret_cast<const float4*>(&ms.o_final[jj][4 * lane]);
                const float4 ob = *reinterpret_cast<const float4*>(&ms.o_final[jb][4 * lane]);
                float va[RP], vb[RP];
#pragma unroll
                for (int ii = 0; ii < RP; ++ii) {
                    va[ii] = fmaf(oa.x, rr[ii].x, fmaf(oa.y, rr[ii].y, fmaf(oa.z, rr[ii].z, oa.w * rr[ii].w)));
                    vb[ii] = fmaf(ob.x, rr[ii].x, fmaf(ob.y, rr[ii].y, fmaf(ob.z, rr[ii].z, ob.w * rr[ii].w)));
                }
                if constexpr (RP == 16) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        va[k] += __shfl_xor_sync(0xffffffffu, va[k], 16);
                        vb[k] += __shfl_xor_sync(0xffffffffu, vb[k], 16);
                    }
                }
#pragma unroll
                for (int off = RP / 2; off >= 1; off >>= 1) {
                    const bool upper = lane & off;
#pragma unroll
                    for (int k = 0; k < off; ++k) {
                        const float sa = upper ? va[k] : va[k + off], ka = upper ? va[k + off] : va[k];
                        const float sb = upper ? vb[k] : vb[k + off], kb = upper ? vb[k + off] : vb[k];
                        va[k] = ka + __shfl_xor_sync(0xffffffffu, sa, off);
                        vb[k] = kb + __shfl_xor_sync(0xffffffffu, sb, off);
                    }
                }
                const int row = RPW * warp + RP * pass + (lane & (RP - 1));
                if (RP == 32 || lane < 16) {
                    const float la = ms.Lh[jj], lb = ms.Lh[jb];
                    const float fa = direct ? (la > 0.f ? 1.f / la : 0.f) : 1.f;
                    const float fb = direct ? (lb > 0.f ? 1.f / lb : 0.f) : 1.f;
                    slot[(size_t)jj * stride + first + row] = va[0] * fa;
                    if (jj + 1 < G) slot[(size_t)(jj + 1) * stride + first + row] = vb[0] * fb;
                }
            }
        }
    }
    if (!direct && tid < G) {
        slot[(size_t)tid * PART_STRIDE] = ms.Mh[tid];
        slot[(size_t)tid * PART_STRIDE + 1] = ms.Lh[tid];
    }
}

// In the last CTA of a unit: merges its n partial slots (slot_of(s), s < n;
// already in the output basis) per head with the log-sum-exp rule and writes
// out[jj][c] = O_c / L (zeros when L = 0) for the G heads.  All threads call
// it.  Each head's partials are spread over P = NW / G warps (split p, p + P,
// ...); a warp loads up to CH of them at once and folds them in with an
// online rescale, so a unit of up to P * CH partials costs one round trip to
// L2; the P per-warp results of a head are then combined in shared memory.
template <int NW, int MAXG, typename SlotFn>
__device__ __forceinline__ void merge_out(MergeSmem<NW, MAXG>& ms, SlotFn slot_of, int n, int G,
                                          float* __restrict__ out) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int CH = 8;  // partials in flight per lane
    const int P = NW / G;  // warps per head (G <= NW)
    float* wo = &ms.red[0][0][0];  // [NW][D] per-warp merged o
    if (warp < P * G) {
        const int jj = warp % G, p = warp / G;
        float M = -CUDART_INF_F, L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = p; s0 < n; s0 += P * CH) {
            float2 ml[CH];
            float4 ov[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int s = s0 + P * k;
                if (s < n) {
                    const float* ph = slot_of(s) + (size_t)jj * PART_STRIDE;
                    ml[k] = __ldcg(reinterpret_cast<const float2*>(ph));
                    ov[k] = ldcg4(ph + 4 + 4 * lane);
                } else {
                    ml[k] = make_float2(-CUDART_INF_F, 0.f);
                    ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const float Mn = fmaxf(M, ml[k].x);
                const float a = Mn == -CUDART_INF_F ? 0.f : ex2(M - Mn);
                const float b = Mn == -CUDART_INF_F ? 0.f : ex2(ml[k].x - Mn);
                L = fmaf(L, a, ml[k].y * b);
                O.x = fmaf(O.x, a, ov[k].x * b);
                O.y = fmaf(O.y, a, ov[k].y * b);
                O.z = fmaf(O.z, a, ov[k].z * b);
                O.w = fmaf(O.w, a, ov[k].w * b);
                M = Mn;
            }
        }
        *reinterpret_cast<float4*>(wo + (size_t)warp * D + 4 * lane) = O;
        if (lane == 0) {
            ms.fac[0][warp] = M;
            ms.lsp[0][warp] = L;
        }
    }
    __syncthreads();
    // combine the P warps of each head and normalise: out = sum_p 2^(M_p - M) O_p / L
    for (int idx = tid; idx < G * (D / 4); idx += NW * 32) {
        const int jj = idx / (D / 4), c4 = idx % (D / 4);
        float M = -CUDART_INF_F;
        for (int p = 0; p < P; ++p) M = fmaxf(M, ms.fac[0][jj + G * p]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < P; ++p) {
            const int w = jj + G * p;
            const float f = M == -CUDART_INF_F ? 0.f : ex2(ms.fac[0][w] - M);
            const float4 v = *reinterpret_cast<const float4*>(wo + (size_t)w * D + 4 * c4);
            L = fmaf(ms.lsp[0][w], f, L);
            O.x = fmaf(v.x, f, O.x);
            O.y = fmaf(v.y, f, O.y);
            O.z = fmaf(v.z, f, O.z);
            O.w = fmaf(v.w, f, O.w);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        *reinterpret_cast<float4*>(out + (size_t)jj * D + 4 * c4) =
            make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
    }
}

}  // namespace kvq
