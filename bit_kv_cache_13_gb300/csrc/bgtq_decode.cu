// Fused decode attention over the packed Block-GTQ cache.
//
// "RoPE-Aware Bit Allocation for KV-Cache Quantization", Figure 2 and core
// method: the kernel reads only the packed code streams and fp16 norms of
// the current tile and decodes them in registers.  Decode works in the TQ
// basis, <q_b, r c Pi^T> = r <q_b Pi, c>: each query sub-vector is rotated
// once per CTA (q~_b = q_b Pi_n), a key contributes r_b C_b[code] q~ per
// coordinate, and values accumulate sum_s p_s r_s C_v[code] in the Pi_128
// basis, rotated back once at the end.
//
// Grid (split, kv_head, seq) with one CTA per SM (12 warps for head groups
// up to 4, 8 for groups of 8); the pages of a (sequence, KV head) are dealt
// round-robin over all warps of its CTAs and streamed through per-warp rings
// of bulk async copies, three pages per mbarrier phase.
//
// Both products run on mma.sync m16n8k16, and their A operands come from
// lookup tables indexed by TWO codes at once, so one shared-memory load
// yields a whole A register (two fp16 elements):
//   QK  K = 16 gathered positions of one width (a chunk; a width group is
//       padded to a multiple of 16 with zero B rows).  Lane t holds the
//       chunk's positions 4t..4t+3, whose 4b code bits are contiguous in a
//       token's stream: positions (4t, 4t+1) are one 2b-bit table index,
//       (4t+2, 4t+3) the next.  For widths up to 5 the key table maps the
//       index to the two scaled centroids as an fp16 hi pair and an fp16 lo
//       pair (about 22 significant bits, one 64-bit load); wider codes use
//       one 32-bit (hi | lo) entry per code.  Rows r and r + 8 of an MMA
//       are the hi and lo parts of one token, so an A quad is two table
//       entries: one MMA covers tokens 0..7, one tokens 8..15.  B = q~ sigma
//       (a per-head power of two) as hi/lo columns.  The MMA accumulators
//       run over a whole width group, and the token's group norm r_{s,b}
//       scales the sum once per group in fp32.
//   softmax  online, base 2, exact running maximum per head; p is rounded to
//       fp16 once (p^), and the same p^ weights the values and the
//       normaliser.
//   PV  rows = channels, K = the 16 tokens of a page.  The value codes of
//       slots 2j and 2j + 1 sit side by side per channel (the tile format),
//       so a (channel, token pair) is one 2 v_bits-bit index into a table of
//       fp16 pairs C_v[c0] / sqrt(128) | C_v[c1] / sqrt(128) << 16: exactly
//       an A register.  Lane (r, t) owns channels 16r .. 16r+15 of token
//       pairs t and t + 4 (v_bits words each).  B = p^ r_v as an exact fp16
//       hi/lo pair in the N columns.
// The tables live in a static shared-memory area; each table is replicated
// across the banks (entry e, copy c at e * copies + c, a lane reads copy
// lane % copies), so a warp's random lookups mostly hit distinct banks, and
// since each table sits at an offset aligned to its size, an entry's offset
// is index | (table offset | copy offset): one LOP3 on the index, which the
// code window already holds at the right bit position.
#include <cmath>
#include <type_traits>
#include <mutex>

#include "bgtq_common.cuh"

namespace kvq {

constexpr int BG_MAX_STAGES = 8;
constexpr int BG_UNIT = 3;  // pages per mbarrier phase (ring stages come in threes)

template <int MAXG>
struct BgWarps {
    static constexpr int NW = MAXG <= 4 ? 12 : 8;
};

// QK works on chunks of 16 gathered positions of one width (a group's
// positions padded to a multiple of 16): at most 64/8 + 7 = 15 chunks.
constexpr int BG_MAX_CHUNKS = 16;
struct BgChunk {
    int16_t b;     // width
    int16_t pos0;  // first gathered position
};

// ---- lookup tables (byte offsets in the table area; each pair table is
// aligned, within the area, to its size)
constexpr int KP_MAX = 5;  // key widths with pair tables
constexpr int VP_MAX = 5;  // value widths with pair tables
// log2 of the copies of each pair table: 16 copies make a half-warp's 64-bit
// lookups (banks 2c, 2c+1) conflict-free, 32 a warp's 32-bit ones
__host__ __device__ constexpr int kp_lg_copies(int b) { return b <= 3 ? 4 : (b == 4 ? 2 : 0); }
__host__ __device__ constexpr int vp_lg_copies(int b) { return b <= 3 ? 5 : (b == 4 ? 3 : 1); }
// key pair table of width b: 4^b entries x copies x 8 bytes, aligned to its size
__host__ __device__ constexpr int kp_off(int b) {
    return b == 3 ? 0 : b == 4 ? 8192 : b == 5 ? 16384 : b == 2 ? 32768 : 34816;
}
constexpr int V_OFF = 24576;   // value table: pairs (4^v x copies x 4 B) or fp16 per code
constexpr int KS_OFF = 35328;  // single-code key tables of widths 6..8: (hi | lo << 16) per code
__host__ __device__ constexpr int ks_off(int b) { return KS_OFF + (b == 6 ? 0 : b == 7 ? 256 : 768); }
constexpr int LUT_BYTES = KS_OFF + 1792;
static_assert((1 << (2 * 1)) * 16 * 8 == 512 && kp_off(1) % 512 == 0 && kp_off(1) + 512 <= KS_OFF, "key table 1");
static_assert((1 << (2 * 2)) * 16 * 8 == 2048 && kp_off(2) % 2048 == 0 && kp_off(2) + 2048 <= kp_off(1), "key table 2");
static_assert((1 << (2 * 3)) * 16 * 8 == 8192 && (1 << (2 * 4)) * 4 * 8 == 8192 && (1 << (2 * 5)) * 8 == 8192,
              "key tables 3..5");
static_assert((1 << (2 * 3)) * 32 * 4 == 8192 && (1 << (2 * 4)) * 8 * 4 == 8192 && (1 << (2 * 5)) * 2 * 4 == 8192,
              "value tables");
static_assert(V_OFF % 8192 == 0 && V_OFF + 8192 <= kp_off(2), "value table place");

// scaled centroids of every width (width b at 2^b - 2) and of the values
constexpr int CBS_V = 510;

// 1 / sqrt(n) for even n = 2i (v[0] unused), computed on the host in fp64
// (correctly rounded, as on the device) and passed with the launch: the
// kernel needs one per width group, and fp64 arithmetic is slow here.
struct RsqrtTab {
    double v[D / 2 + 1];
};

template <int NW, int MAXG>
struct __align__(16) BgDecodeSmem {
    uint2 bfr[BG_MAX_CHUNKS][MAXG / 4][32];  // QK B fragments per chunk, n-tile and lane
    float cbs[CBS_V + 256];                  // fp32(C_b / sqrt(n_b)) per width, then fp32(C_v / sqrt(128))
    double rsn[9];                           // 1 / sqrt(n): [0] values (n = 128), [b] the width-b group
    BgChunk chunks[BG_MAX_CHUNKS];
    int n_chunks;
    float sigma[MAXG];      // power-of-two pre-scale per head
    __half pbh[NW][MAXG][BG_UNIT * PAGE];  // p^ of the warp's current unit, head-major
    float qt[MAXG][D];         // q~ in gathered order, times scale * log2(e)
    float qin[MAXG][D];
    uint64_t bar[NW][BG_MAX_STAGES];
    int ntok[NW][BG_MAX_STAGES];
    BgtqLayout L;
    int kbase[9], nch[9];   // first chunk and chunk count of each width
    int64_t pioff[D / 2 + 1];  // offset of Pi_n (n = 2i) in the rotation table
    float qpart[NW * 32 / D - 1][MAXG][D];  // partial q~ sums of the other thread groups
    int8_t wsm[D / 2];      // this head's block widths
    MergeSmem<NW, MAXG> ms;
};

template <int N>
__device__ __forceinline__ uint32_t shift_left(uint32_t x) {
    if constexpr (N >= 0)
        return x << N;
    else
        return x >> (-N);
}

__device__ __forceinline__ uint32_t pack_hi_lo(float v, bool lo) {
    const __half h = __float2half_rn(v);
    return lo ? (uint32_t)__half_as_ushort(__float2half_rn(v - __half2float(h))) : (uint32_t)__half_as_ushort(h);
}

// Fill the tables of this head (every thread of the CTA; the scaled
// centroids are in cbs, and a barrier follows).  The key tables only with
// valid widths (keys: the present widths); the value table always, so that
// nothing reads uninitialised shared memory.
template <int VB>
__device__ __forceinline__ void build_tables(uint8_t* lut, const float* cbs, const BgtqLayout& L, int nthreads,
                                             bool keys) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int b = 1; b <= KP_MAX; ++b) {
        if (!keys || L.n[b] == 0) continue;
        const int lg = kp_lg_copies(b), cnt = (1 << (2 * b)) << lg;
        const float* cb = cbs + (1 << b) - 2;
        uint2* tab = reinterpret_cast<uint2*>(lut + kp_off(b));
        for (int idx = tid; idx < cnt; idx += nthreads) {
            const int e = idx >> lg, c0 = e & ((1 << b) - 1), c1 = e >> b;
            const float v0 = cb[c0], v1 = cb[c1];
            tab[idx] = make_uint2(pack_hi_lo(v0, false) | (pack_hi_lo(v1, false) << 16),
                                  pack_hi_lo(v0, true) | (pack_hi_lo(v1, true) << 16));
        }
    }
#pragma unroll
    for (int b = KP_MAX + 1; b <= 8; ++b) {
        if (!keys || L.n[b] == 0) continue;
        const float* cb = cbs + (1 << b) - 2;
        uint32_t* tab = reinterpret_cast<uint32_t*>(lut + ks_off(b));
        for (int c = tid; c < (1 << b); c += nthreads) tab[c] = pack_hi_lo(cb[c], false) | (pack_hi_lo(cb[c], true) << 16);
    }
    const float* cv = cbs + CBS_V;
    if constexpr (VB <= VP_MAX) {
        constexpr int lg = vp_lg_copies(VB), cnt = (1 << (2 * VB)) << lg;
        uint32_t* tab = reinterpret_cast<uint32_t*>(lut + V_OFF);
        for (int idx = tid; idx < cnt; idx += nthreads) {
            const int e = idx >> lg, c0 = e & ((1 << VB) - 1), c1 = e >> VB;
            tab[idx] = (uint32_t)__half_as_ushort(__float2half_rn(cv[c0])) |
                       ((uint32_t)__half_as_ushort(__float2half_rn(cv[c1])) << 16);
        }
    } else {
        __half* tab = reinterpret_cast<__half*>(lut + V_OFF);
        for (int c = tid; c < (1 << VB); c += nthreads) tab[c] = __float2half_rn(cv[c]);
    }
}

// D = A B (+ 0): the first MMA of an accumulator needs no zeroed registers.
__device__ __forceinline__ void mma_f16_16816_first(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// Bits the lane's code window is shifted left by before the lookups: the
// first position pair then sits where the table index goes.
template <int B>
__host__ __device__ constexpr int qk_pre_shift() { return B <= KP_MAX ? 3 + kp_lg_copies(B) : 0; }

// QK of one chunk (16 positions of width B) for the unit's pages: the MMA
// accumulators cg run over the chunk's width group (FIRST: the group's first
// chunk starts them).  xw: per page, the lane's 4B code bits of tokens r and
// r + 8, shifted left by qk_pre_shift<B>() (garbage below).  tsel: the byte
// offset of the lane's copy of the width's table in the table area (the
// table is aligned to its size, so an entry's offset is index | tsel).
template <int B, int NT, bool FIRST>
__device__ __forceinline__ void qk_chunk(const uint32_t (&xw)[BG_UNIT][2], uint32_t tsel, const uint2 (&bb)[NT],
                                         float (&cg)[2][BG_UNIT][NT][4], const uint8_t* __restrict__ lut) {
#pragma unroll
    for (int e = 0; e < BG_UNIT; ++e) {
        const uint32_t x0 = xw[e][0], x8 = xw[e][1];
        // Two MMAs per page: rows r / r + 8 of the first are token r's hi /
        // lo centroid parts, of the second token r + 8's, so each A quad is
        // two table entries (hi pair, lo pair) of one token: positions
        // (4t, 4t+1) give a0, a1 and positions (4t+2, 4t+3) give a2, a3.
        uint32_t aA[4], aB[4];
        if constexpr (B <= KP_MAX) {
            constexpr int S = qk_pre_shift<B>();
            constexpr uint32_t MK = ((1u << (2 * B)) - 1u) << S;
            const uint2 e0 = *reinterpret_cast<const uint2*>(lut + ((x0 & MK) | tsel));
            const uint2 e2 = *reinterpret_cast<const uint2*>(lut + (((x0 >> (2 * B)) & MK) | tsel));
            const uint2 e1 = *reinterpret_cast<const uint2*>(lut + ((x8 & MK) | tsel));
            const uint2 e3 = *reinterpret_cast<const uint2*>(lut + (((x8 >> (2 * B)) & MK) | tsel));
            aA[0] = e0.x; aA[1] = e0.y; aA[2] = e2.x; aA[3] = e2.y;
            aB[0] = e1.x; aB[1] = e1.y; aB[2] = e3.x; aB[3] = e3.y;
        } else {
            constexpr uint32_t M = (1u << B) - 1u;
#pragma unroll
            for (int j = 0; j < 2; ++j) {  // position pair j of the lane: codes at bits 2jB, (2j+1)B
                const uint32_t* tab = reinterpret_cast<const uint32_t*>(lut + tsel);
                const uint32_t c0 = tab[(x0 >> (2 * j * B)) & M], c1 = tab[(x0 >> ((2 * j + 1) * B)) & M];
                const uint32_t d0 = tab[(x8 >> (2 * j * B)) & M], d1 = tab[(x8 >> ((2 * j + 1) * B)) & M];
                aA[2 * j] = prmt(c0, c1, 0x5410);
                aA[2 * j + 1] = prmt(c0, c1, 0x7632);
                aB[2 * j] = prmt(d0, d1, 0x5410);
                aB[2 * j + 1] = prmt(d0, d1, 0x7632);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {  // tokens r and r + 8 in separate chains
            if constexpr (FIRST) {
                mma_f16_16816_first(cg[0][e][nt], aA, bb[nt].x, bb[nt].y);
                mma_f16_16816_first(cg[1][e][nt], aB, bb[nt].x, bb[nt].y);
            } else {
                mma_f16_16816(cg[0][e][nt], aA, bb[nt].x, bb[nt].y);
                mma_f16_16816(cg[1][e][nt], aB, bb[nt].x, bb[nt].y);
            }
        }
    }
}

// QK of the unit's pages over every chunk of width B (all in registers but
// the B fragments), then the group norm r_{s,B} of each token scales the
// group's dot products once, in fp32.
template <int B, int NT, int NW, int MAXG>
__device__ __forceinline__ void qk_width(const uint8_t* const (&tiles)[BG_UNIT], const BgtqTile& tl, int lane,
                                         const BgDecodeSmem<NW, MAXG>& sm, float (&acc)[BG_UNIT][NT][2],
                                         const uint8_t* __restrict__ lut) {
    const int nch = sm.nch[B];
    if (nch == 0) return;  // warp-uniform
    const int r = lane >> 2, t = lane & 3, k0 = sm.kbase[B];
    constexpr int S = qk_pre_shift<B>();
    uint32_t tsel;
    if constexpr (B <= KP_MAX)
        tsel = kp_off(B) | (((uint32_t)lane << 3) & ((1u << S) - 1u));  // the lane's copy
    else
        tsel = ks_off(B);
    float cg[2][BG_UNIT][NT][4];
    // the window starts S bits before the lane's first code bit (for the
    // stream's first bit that is inside the word before it: the previous
    // token's record, or the shared memory below the ring; those bits are
    // masked off)
    int off = sm.L.bitstart[B] + 4 * t * B - S;
    auto chunk = [&](int c, auto first) {
        uint2 bb[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) bb[nt] = sm.bfr[k0 + c][nt][lane];
        const int wofs = (off >> 5) * 4, sh = off & 31;
        uint32_t xw[BG_UNIT][2];
#pragma unroll
        for (int e = 0; e < BG_UNIT; ++e)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(tiles[e] + (r + 8 * i) * tl.kb + wofs);
                xw[e][i] = __funnelshift_r(w[0], w[1], sh);
            }
        qk_chunk<B, NT, decltype(first)::value>(xw, tsel, bb, cg, lut);
        off += 16 * B;
    };
    chunk(0, std::true_type{});
#pragma unroll 1
    for (int c = 1; c < nch; ++c) chunk(c, std::false_type{});
#pragma unroll
    for (int e = 0; e < BG_UNIT; ++e) {
        const __half* nrm = reinterpret_cast<const __half*>(tiles[e] + tl.off_kn + 2 * (B - 1));
        const float rn0 = __half2float(nrm[8 * r]), rn8 = __half2float(nrm[8 * (r + 8)]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // rows r (hi) and r + 8 (lo) of each MMA, columns q~ hi and lo
            const float s0 = (cg[0][e][nt][0] + cg[0][e][nt][1]) + (cg[0][e][nt][2] + cg[0][e][nt][3]);
            const float s8 = (cg[1][e][nt][0] + cg[1][e][nt][1]) + (cg[1][e][nt][2] + cg[1][e][nt][3]);
            acc[e][nt][0] = fmaf(rn0, s0, acc[e][nt][0]);
            acc[e][nt][1] = fmaf(rn8, s8, acc[e][nt][1]);
        }
    }
}

// The table entry (an A register) of channel 16r + I of the lane's field f
// (the v_bits words of one token pair); vsel: the byte offset of the lane's
// copy of the value table in the table area.
template <int VB, int I>
__device__ __forceinline__ uint32_t v_entry(const uint32_t (&f)[VB], uint32_t vsel, const uint8_t* __restrict__ lut) {
    constexpr int BIT = 2 * VB * I, W = BIT >> 5, SH = BIT & 31;
    constexpr bool STRADDLE = SH + 2 * VB > 32;
    if constexpr (VB <= VP_MAX) {
        constexpr int SV = 2 + vp_lg_copies(VB);
        constexpr uint32_t MV = ((1u << (2 * VB)) - 1u) << SV;
        uint32_t x;
        if constexpr (STRADDLE)
            x = __funnelshift_r(f[W], f[W + 1], SH - SV);  // SH > 32 - 2 VB >= SV here
        else
            x = shift_left<SV - SH>(f[W]);
        return *reinterpret_cast<const uint32_t*>(lut + ((x & MV) | vsel));
    } else {
        constexpr uint32_t M = (1u << VB) - 1u;
        uint32_t x;
        if constexpr (STRADDLE)
            x = __funnelshift_r(f[W], f[W + 1], SH);
        else
            x = f[W] >> SH;
        const unsigned short* tab = reinterpret_cast<const unsigned short*>(lut + vsel);
        return (uint32_t)tab[x & M] | ((uint32_t)tab[(x >> VB) & M] << 16);
    }
}

// PV of one page: oacc[m] += A(channels 16r + 2m, 16r + 2m + 1 x the 16
// tokens) B(p^ r_v hi, lo).
template <int VB, int NT>
__device__ __forceinline__ void pv_page(const uint8_t* tile, int off_vc, int lane, uint32_t bh0, uint32_t bh1,
                                        uint32_t bl0, uint32_t bl1, float (&oacc)[8][4],
                                        const uint8_t* __restrict__ lut) {
    const int r = lane >> 2, t = lane & 3;
    const uint32_t* p0 = reinterpret_cast<const uint32_t*>(tile + off_vc + 32 * VB * t + 4 * VB * r);
    const uint32_t* p1 = reinterpret_cast<const uint32_t*>(tile + off_vc + 32 * VB * (t + 4) + 4 * VB * r);
    uint32_t f0[VB], f1[VB];
#pragma unroll
    for (int w = 0; w < VB; ++w) {
        f0[w] = p0[w];
        f1[w] = p1[w];
    }
    // the lane's copy of the value table (the table is aligned to its size)
    uint32_t vsel = V_OFF;
    if constexpr (VB <= VP_MAX) vsel |= ((uint32_t)lane << 2) & ((1u << (2 + vp_lg_copies(VB))) - 1u);
    // a0 = (channel 16r + 2m, tokens 2t, 2t+1), a1 = (16r + 2m + 1, same),
    // a2 = (16r + 2m, tokens 2t+8, 2t+9), a3 = (16r + 2m + 1, same)
#define KVQ_PV_M(m)                                                                                   \
    {                                                                                                 \
        const uint32_t a[4] = {v_entry<VB, 2 * (m)>(f0, vsel, lut), v_entry<VB, 2 * (m) + 1>(f0, vsel, lut),   \
                               v_entry<VB, 2 * (m)>(f1, vsel, lut), v_entry<VB, 2 * (m) + 1>(f1, vsel, lut)}; \
        mma_f16_16816(oacc[m], a, bh0, bh1);                                                          \
        if constexpr (NT == 2) mma_f16_16816(oacc[m], a, bl0, bl1);                                   \
    }
    KVQ_PV_M(0) KVQ_PV_M(1) KVQ_PV_M(2) KVQ_PV_M(3) KVQ_PV_M(4) KVQ_PV_M(5) KVQ_PV_M(6) KVQ_PV_M(7)
#undef KVQ_PV_M
}

// ---- kernel body follows

template <int MAXG, int VB>
__global__ void __launch_bounds__(BgWarps<MAXG>::NW * 32, 1)
bgtq_decode_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int G, const uint8_t* __restrict__ cache,
                   int64_t num_pages, const int32_t* __restrict__ block_table, int max_pages,
                   const int32_t* __restrict__ context_lens, const int8_t* __restrict__ widths, int total_bits,
                   int v_bits, const float* __restrict__ pi_table, const int64_t* __restrict__ pi_offsets,
                   const double* __restrict__ codebooks, float scale_log2, float* __restrict__ out,
                   uint8_t* __restrict__ ws, int n_stages, const RsqrtTab rs) {
    constexpr int NW = BgWarps<MAXG>::NW;
    constexpr int NT = MAXG / 4;  // n-tiles of 8 columns (4 heads x hi/lo)
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ __align__(16) uint8_t lut[LUT_BYTES];
    BgDecodeSmem<NW, MAXG>& sm = *reinterpret_cast<BgDecodeSmem<NW, MAXG>*>(smem_raw);
    const BgtqTile tl(total_bits, VB);
    // the page rings follow the fixed part; after the loop the per-warp o'
    // partials take their place (the host sizes the region for both)
    uint8_t* ring_base = smem_raw + align_up(sizeof(BgDecodeSmem<NW, MAXG>), 128);
    uint8_t* my_ring = ring_base + (size_t)(threadIdx.x >> 5) * n_stages * tl.bytes;
    float(*o_part)[MAXG][D] = reinterpret_cast<float(*)[MAXG][D]>(ring_base);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int S = gridDim.x, B = gridDim.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* err_word = reinterpret_cast<uint32_t*>(ws);

    {
        // prefetches into L2 only (coherent with any later write of the
        // previous kernel): the warp's first block-table entries, the
        // context length, the query rows and the output rotation
        const int j = split * NW + warp + S * NW * lane;
        if (lane <= BG_MAX_STAGES && j < max_pages) prefetch_l2(block_table + (size_t)b * max_pages + j);
        if (tid == 0) prefetch_l2(context_lens + b);
        const char* qc = reinterpret_cast<const char*>(q + ((size_t)b * H_q + (size_t)h * G) * D);
        if (tid < (G * D * 2 + 127) / 128) prefetch_l2(qc + 128 * tid);
    }
    griddep_wait();  // every input may come from the previous kernel in the stream
    // ---- every small input is requested in one round trip, before any page
    // copy (under the page stream a read waits microseconds behind the
    // copies): the context length, the warp's first block-table entries
    // (bounded by the table row, checked against the length later), the
    // widths, the rotation offsets, the query rows and every codebook entry
    // a width could use.
    constexpr int NTHR = NW * 32;
    const int32_t* bt = block_table + (size_t)b * max_pages;
    // pages dealt round-robin over all S * NW warps of the (sequence, KV head)
    const int KS = S * NW, k0 = split * NW + warp;
    auto page_of = [&](int j) { return k0 + KS * j; };
    const int ctx_in = __ldg(context_lens + b);
    int pid_pre[BG_MAX_STAGES / BG_UNIT + 1];
#pragma unroll
    for (int u = 0; u <= BG_MAX_STAGES / BG_UNIT; ++u) {
        const int pg = page_of(BG_UNIT * u + lane);
        pid_pre[u] = lane < BG_UNIT && u <= n_stages / BG_UNIT && pg < max_pages ? __ldg(bt + pg) : 0;
    }
    if (tid < D / 2) sm.wsm[tid] = __ldg(widths + h * (D / 2) + tid);
    if (tid <= D / 2) sm.pioff[tid] = __ldg(pi_offsets + 2 * tid);  // Pi_n for even n = 2 tid
    {
        const uint4* q4 = reinterpret_cast<const uint4*>(q + ((size_t)b * H_q + (size_t)h * G) * D);
        const int nq4 = G * D / 8, i4 = tid - D / 2;
        if (i4 >= 0 && i4 < nq4) {  // 8 bf16 per thread
            const uint4 w = __ldg(q4 + i4);
            const __nv_bfloat16* e8 = reinterpret_cast<const __nv_bfloat16*>(&w);
#pragma unroll
            for (int k = 0; k < 8; ++k) sm.qin[(8 * i4 + k) / D][(8 * i4 + k) % D] = __bfloat162float(e8[k]);
        }
    }
    // codebook entries: thread slot j < CBS_V + 2^VB holds entry j in a register
    // until the group sizes are known (width b code c at 2^b - 2 + c)
    double craw[(CBS_V + 256 + NTHR - 1) / NTHR];
#pragma unroll
    for (int u = 0; u < (CBS_V + 256 + NTHR - 1) / NTHR; ++u) {
        const int idx = tid + u * NTHR;
        craw[u] = 0.0;
        if (idx < CBS_V) {
            const int bb = 31 - __clz(idx + 2), c = idx + 2 - (1 << bb);
            craw[u] = __ldg(codebooks + (bb - 1) * 256 + c);
        } else if (idx < CBS_V + (1 << VB)) {
            craw[u] = __ldg(codebooks + (VB - 1) * 256 + idx - CBS_V);
        }
    }
    const int ctx = max(0, min(ctx_in, max_pages * PAGE));
    const int n_pages = (ctx + PAGE - 1) / PAGE;
    const int my_count = n_pages > k0 ? (n_pages - k0 + KS - 1) / KS : 0;

    // Pages travel in units of BG_UNIT (one mbarrier phase, one wait, one
    // release): unit u is the warp's pages BG_UNIT u .. + BG_UNIT - 1 in the
    // ring slots of slot group u % n_grp.
    const int n_grp = n_stages / BG_UNIT;
    const int n_units = (my_count + BG_UNIT - 1) / BG_UNIT;
    if (lane == 0) {
        for (int s = 0; s < n_grp; ++s) mbar_init(&sm.bar[warp][s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    auto issue_unit = [&](int u, int st, int pid) {
        // whole warp; lane e < BG_UNIT issues page e of unit u (id pid)
        uint64_t* bar = &sm.bar[warp][st];
        const int j = BG_UNIT * u + lane;
        bool ok = false;
        if (lane < BG_UNIT) {
            int n = 0;
            if (j < my_count) {
                if (pid < 0 || (int64_t)pid >= num_pages) {
                    atomicOr(err_word, ERR_BAD_PAGE);
                } else {
                    ok = true;
                    n = min(PAGE, ctx - page_of(j) * PAGE);
                }
            }
            sm.ntok[warp][BG_UNIT * st + lane] = n;
        }
        const uint32_t n_ok = __popc(__ballot_sync(0xffffffffu, ok));
        __syncwarp();  // the lanes' counts are ordered before lane 0's arrive (release)
        if (lane == 0) {
            if (n_ok == 0)
                mbar_arrive(bar);
            else
                mbar_arrive_expect_tx(bar, n_ok * (uint32_t)tl.bytes);
        }
        __syncwarp();  // the expected bytes are set before any copy is issued
        if (ok)
            bulk_g2s(my_ring + (size_t)(BG_UNIT * st + lane) * tl.bytes, cache + ((size_t)pid * H_kv + h) * tl.bytes,
                     tl.bytes, bar);
    };
    // the first slot group's copies now; the others once the setup's own
    // reads are out (below)
    int pid_next = 0, n_issued = 0;
    if (n_units > 0) {  // warp-uniform
        issue_unit(0, 0, pid_pre[0]);
        n_issued = 1;
    }
#pragma unroll
    for (int u = 0; u <= BG_MAX_STAGES / BG_UNIT; ++u)
        if (u == n_grp) pid_next = pid_pre[u];
    {
        // the block table is read later: have L2 keep it
        const char* btc = reinterpret_cast<const char*>(bt);
        const int lines = (n_pages * 4 + 127) / 128;
        for (int l = split * NW * 32 + tid; l < lines; l += S * NW * 32) prefetch_l2_keep(btc + 128 * l);
    }

    // ---- per-head layout, chunk schedule, tables and rotated queries
    __syncthreads();
    {
        // the output rotation is read at the end: have L2 keep it
        const char* rot = reinterpret_cast<const char*>(pi_table + sm.pioff[D / 2]);
        for (int l = tid; l < D * D * 4 / 128; l += NTHR) prefetch_l2_keep(rot + 128 * l);
    }
    if (warp == 0) {
        // the layout by ballots: groups by ascending width, blocks ascending
        // in a group, block i as (dim i, dim i + 64); then the chunk list and
        // 1 / sqrt(n) per group (fp64, once)
        const int w0 = sm.wsm[lane], w1 = sm.wsm[lane + 32];
        const bool ok = __all_sync(0xffffffffu, w0 >= 1 && w0 <= 8 && w1 >= 1 && w1 <= 8);
        const uint32_t lt = (1u << lane) - 1u;
        int pos = 0, bit = 0, nc = 0;
#pragma unroll
        for (int bb = 1; bb <= 8; ++bb) {
            const uint32_t m0 = __ballot_sync(0xffffffffu, w0 == bb), m1 = __ballot_sync(0xffffffffu, w1 == bb);
            const int cnt = __popc(m0) + __popc(m1);
            if (w0 == bb) {
                const int rk = __popc(m0 & lt);
                sm.L.dim[pos + 2 * rk] = (int16_t)lane;
                sm.L.dim[pos + 2 * rk + 1] = (int16_t)(lane + D / 2);
            }
            if (w1 == bb) {
                const int rk = __popc(m0) + __popc(m1 & lt);
                sm.L.dim[pos + 2 * rk] = (int16_t)(lane + 32);
                sm.L.dim[pos + 2 * rk + 1] = (int16_t)(lane + 32 + D / 2);
            }
            const int n = 2 * cnt, nch = (n + 15) / 16;
            if (lane == 0) {
                sm.L.start[bb] = (int16_t)pos;
                sm.L.bitstart[bb] = (int16_t)bit;
                sm.L.n[bb] = (int16_t)n;
                sm.kbase[bb] = nc;
                sm.nch[bb] = nch;
            }
            if (lane < nch && nc + lane < BG_MAX_CHUNKS) {
                BgChunk ch;
                ch.b = (int16_t)bb;
                ch.pos0 = (int16_t)(pos + 16 * lane);
                sm.chunks[nc + lane] = ch;
            }
            if (lane == bb) sm.rsn[bb] = rs.v[n / 2];
            pos += n;
            bit += bb * n;
            nc += nch;
        }
        if (lane == 0) {
            sm.L.start[0] = sm.L.n[0] = sm.L.bitstart[0] = 0;
            sm.L.total_bits = bit;
            sm.L.ok = ok && pos == D && nc <= BG_MAX_CHUNKS;
            sm.n_chunks = nc;
            sm.rsn[0] = rs.v[D / 2];
        }
    }
    __syncthreads();
    // the table area must sit on its alignment for the OR-formed addresses
    const bool layout_ok = sm.L.ok && sm.L.total_bits <= 2 * total_bits;
    if (tid == 0 && !layout_ok) atomicOr(err_word, ERR_BAD_WIDTHS);
    // q~ at gathered position p: sum_i q[dim(st + i)] Pi_n[i][p - st], the i
    // split over NPART thread groups (their loads go out together)
    constexpr int NPART = NTHR / D;
    {
        const int p = tid % D, part = tid / D;
        float acc[MAXG];
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) acc[jj] = 0.f;
        int bb = 1;
        while (bb < 8 && !(p >= sm.L.start[bb] && p < sm.L.start[bb] + sm.L.n[bb])) ++bb;
        const int st = sm.L.start[bb], n = layout_ok ? sm.L.n[bb] : 0, j = p - st;
        const float* pi = pi_table + (n > 0 ? sm.pioff[n / 2] : 0);  // (n = 0: nothing is read)
        // the first QROT_REG terms' rotation entries are requested before
        // the later page copies go out, so they do not queue behind them
        constexpr int QROT_REG = 16;
        float pvr[QROT_REG];
#pragma unroll
        for (int k = 0; k < QROT_REG; ++k) {
            const int i = part + NPART * k;
            pvr[k] = i < n ? __ldg(pi + (size_t)i * n + j) : 0.f;
        }
        // the page copies of the remaining slot groups
#pragma unroll
        for (int u = 1; u < BG_MAX_STAGES / BG_UNIT; ++u)
            if (u < n_grp && u < n_units) {  // warp-uniform
                issue_unit(u, u, pid_pre[u]);
                n_issued = u + 1;
            }
#pragma unroll
        for (int k = 0; k < QROT_REG; ++k) {
            const int i = part + NPART * k;
            if (i < n) {
                const int dm = sm.L.dim[st + i];
#pragma unroll
                for (int jj = 0; jj < MAXG; ++jj)
                    if (jj < G) acc[jj] = fmaf(sm.qin[jj][dm], pvr[k], acc[jj]);
            }
        }
#pragma unroll 8
        for (int i = part + NPART * QROT_REG; i < n; i += NPART) {  // groups of more than 48 (or 32) positions
            const float pv = __ldg(pi + (size_t)i * n + j);
            const int dm = sm.L.dim[st + i];
#pragma unroll
            for (int jj = 0; jj < MAXG; ++jj)
                if (jj < G) acc[jj] = fmaf(sm.qin[jj][dm], pv, acc[jj]);
        }
        if (part > 0) {
#pragma unroll
            for (int jj = 0; jj < MAXG; ++jj) sm.qpart[part - 1][jj][p] = acc[jj];
        }
        // scaled centroids fp32(C_b[c] / sqrt(n_b)) from the registers
#pragma unroll
        for (int u = 0; u < (CBS_V + 256 + NTHR - 1) / NTHR; ++u) {
            const int idx = tid + u * NTHR;
            if (idx < CBS_V) {
                const int bb = 31 - __clz(idx + 2);
                sm.cbs[idx] = __double2float_rn(craw[u] * sm.rsn[bb]);
            } else if (idx < CBS_V + (1 << VB)) {
                sm.cbs[idx] = __double2float_rn(craw[u] * sm.rsn[0]);
            }
        }
        __syncthreads();
        if (part == 0) {
#pragma unroll
            for (int k = 0; k < NPART - 1; ++k)
#pragma unroll
                for (int jj = 0; jj < MAXG; ++jj) acc[jj] += sm.qpart[k][jj][p];
#pragma unroll
            for (int jj = 0; jj < MAXG; ++jj) sm.qt[jj][p] = jj < G ? acc[jj] * scale_log2 : 0.f;
        }
    }
    build_tables<VB>(lut, sm.cbs, sm.L, NTHR, layout_ok);
    __syncthreads();
    // per head: power-of-two pre-scale so that max |q~| sigma is in [2^14, 2^15)
    for (int jj = warp; jj < MAXG; jj += NW) {
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) mx = fmaxf(mx, fabsf(sm.qt[jj][32 * k + lane]));
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) sm.sigma[jj] = mx > 0.f ? ldexpf(1.f, 14 - ilogbf(mx)) : 1.f;
    }
    __syncthreads();

    const int r = lane >> 2, t = lane & 3;
    // ---- QK B fragments: column n = r -> head 4 nt + (r >> 1), part r & 1
    // (hi / lo of q~ sigma); rows k = 2t, 2t+1 (b0) are the chunk positions
    // 4t, 4t+1 and k = 2t+8, 2t+9 (b1) the positions 4t+2, 4t+3, so a lane's
    // two position pairs are adjacent in the code stream; positions past the
    // group are zero
    const int NC = layout_ok ? sm.n_chunks : 0;
    for (int idx = warp; idx < NC * NT; idx += NW) {
        const int k = idx / NT, nt = idx % NT;
        const BgChunk ch = sm.chunks[k];
        const int hq = 4 * nt + (r >> 1), gend = sm.L.start[ch.b] + sm.L.n[ch.b];
        uint32_t w[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int p = ch.pos0 + 4 * t + 2 * e + u;
                v[u] = (hq < G && p < gend) ? sm.qt[hq][p] * sm.sigma[hq] : 0.f;
            }
            const __half h0 = __float2half_rn(v[0]), h1 = __float2half_rn(v[1]);
            w[e] = (r & 1) ? pack_half2(v[0] - __half2float(h0), v[1] - __half2float(h1))
                           : h2_as_u32(__halves2half2(h0, h1));
        }
        sm.bfr[k][nt][lane] = make_uint2(w[0], w[1]);
    }
    float inv_sig[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) inv_sig[nt] = 4 * nt + t < G ? 1.f / sm.sigma[4 * nt + t] : 0.f;
    __syncthreads();  // the tables and B fragments are complete

    // PV accumulators: chunk m, C fragment (row r, r + 8 = channels 16r + 2m,
    // 16r + 2m + 1; columns 2t, 2t + 1)
    float oacc[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[m][e] = 0.f;
    // online softmax state of head 4 nt + t
    float mrun[NT], lsum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrun[nt] = -CUDART_INF_F;
        lsum[nt] = 0.f;
    }
    int u_fail = -1;  // the unit whose wait timed out
    int st = 0;             // u % n_grp
    uint32_t parity = 0u;   // (u / n_grp) & 1

    for (int u = 0; u < n_units; ++u) {
        const bool ok = mbar_wait_bounded(&sm.bar[warp][st], parity, WAIT_LIMIT_CYCLES);
        if (__any_sync(0xffffffffu, !ok)) {
            u_fail = u;
            if (lane == 0) atomicOr(err_word, ERR_TIMEOUT);
            break;
        }
        const uint8_t* tiles[BG_UNIT];
        int n_tok[BG_UNIT];
#pragma unroll
        for (int e = 0; e < BG_UNIT; ++e) {
            tiles[e] = my_ring + (size_t)(BG_UNIT * st + e) * tl.bytes;
            n_tok[e] = layout_ok ? sm.ntok[warp][BG_UNIT * st + e] : 0;
        }

        // ---- QK on the tensor cores, width by width for the unit's pages
        float lg[BG_UNIT][NT][2];
        {
            float acc[BG_UNIT][NT][2];
#pragma unroll
            for (int e = 0; e < BG_UNIT; ++e)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[e][nt][0] = acc[e][nt][1] = 0.f;
            if (NC > 0) {  // warp-uniform
                qk_width<1, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<2, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<3, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<4, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<5, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<6, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<7, NT>(tiles, tl, lane, sm, acc, lut);
                qk_width<8, NT>(tiles, tl, lane, sm, acc, lut);
            }
#pragma unroll
            for (int e = 0; e < BG_UNIT; ++e)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    lg[e][nt][0] = r < n_tok[e] ? acc[e][nt][0] * inv_sig[nt] : -CUDART_INF_F;
                    lg[e][nt][1] = r + 8 < n_tok[e] ? acc[e][nt][1] * inv_sig[nt] : -CUDART_INF_F;
                }
        }

        // ---- online softmax (base 2) of head 4 nt + t; p^ goes to pbh
        float corr[NT];
        bool need = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float pm = fmaxf(lg[0][nt][0], lg[0][nt][1]);
#pragma unroll
            for (int e = 1; e < BG_UNIT; ++e) pm = fmaxf(pm, fmaxf(lg[e][nt][0], lg[e][nt][1]));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
            corr[nt] = 1.f;
            if (pm > mrun[nt]) {
                corr[nt] = ex2(mrun[nt] - pm);
                mrun[nt] = pm;
                need = true;
            }
            const float mref = mrun[nt] == -CUDART_INF_F ? 0.f : mrun[nt];
            float ps = 0.f;
            const int hq = 4 * nt + t;
#pragma unroll
            for (int e = 0; e < BG_UNIT; ++e) {
                const __half p0 = __float2half_rn(ex2(lg[e][nt][0] - mref));
                const __half p8 = __float2half_rn(ex2(lg[e][nt][1] - mref));
                ps += __half2float(p0) + __half2float(p8);
                if (hq < MAXG) {
                    sm.pbh[warp][hq][PAGE * e + r] = p0;
                    sm.pbh[warp][hq][PAGE * e + r + 8] = p8;
                }
            }
            lsum[nt] = fmaf(lsum[nt], corr[nt], ps);
        }
        if (__any_sync(0xffffffffu, need)) {
            // PV columns 2t, 2t + 1: heads (2t) & 3, (2t + 1) & 3 for groups up
            // to 4 (columns 4..7 hold the low parts), heads 2t, 2t + 1 for 8;
            // head h's correction lives in lane h & 3, n-tile h >> 2
            const int hA = 2 * t, hB = 2 * t + 1;
            float cA = __shfl_sync(0xffffffffu, corr[0], hA & 3), cB = __shfl_sync(0xffffffffu, corr[0], hB & 3);
            if constexpr (NT == 2) {
                const float cA1 = __shfl_sync(0xffffffffu, corr[1], hA & 3);
                const float cB1 = __shfl_sync(0xffffffffu, corr[1], hB & 3);
                if (hA >= 4) cA = cA1;
                if (hB >= 4) cB = cB1;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                oacc[m][0] *= cA;
                oacc[m][2] *= cA;
                oacc[m][1] *= cB;
                oacc[m][3] *= cB;
            }
        }
        __syncwarp();

        // ---- PV: B = p^ r_v for column n = r (head r & 3, hi for r < 4 and
        // lo for r >= 4; head r, hi then lo, for groups of 8); rows k =
        // tokens 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1).  Slots past the context
        // get r_v = 0 (their p^ is 0, but a stale norm may be NaN).
#pragma unroll
        for (int e = 0; e < BG_UNIT; ++e) {
            const uint8_t* tile = tiles[e];
            const bool full = n_tok[e] == PAGE;
            const int hq = NT == 1 ? (r & 3) : r;
            const uint32_t* vn = reinterpret_cast<const uint32_t*>(tile + tl.off_vn);
            uint32_t R0 = vn[t], R1 = vn[t + 4];
            if (!full) {
                const uint32_t lo16 = 0x0000ffffu, hi16 = 0xffff0000u;
                R0 &= (2 * t < n_tok[e] ? lo16 : 0u) | (2 * t + 1 < n_tok[e] ? hi16 : 0u);
                R1 &= (2 * t + 8 < n_tok[e] ? lo16 : 0u) | (2 * t + 9 < n_tok[e] ? hi16 : 0u);
            }
            uint32_t P0 = 0u, P1 = 0u;
            if (hq < G) {
                P0 = lds32(&sm.pbh[warp][hq][PAGE * e + 2 * t]);
                P1 = lds32(&sm.pbh[warp][hq][PAGE * e + 2 * t + 8]);
            }
            const __half2 H0 = __hmul2(u32_as_h2(P0), u32_as_h2(R0)), H1 = __hmul2(u32_as_h2(P1), u32_as_h2(R1));
            const __half2 L0 = __hfma2(u32_as_h2(P0), u32_as_h2(R0), __hneg2(H0));
            const __half2 L1 = __hfma2(u32_as_h2(P1), u32_as_h2(R1), __hneg2(H1));
            uint32_t bh0 = h2_as_u32(H0), bh1 = h2_as_u32(H1), bl0 = h2_as_u32(L0), bl1 = h2_as_u32(L1);
            if constexpr (NT == 1) {
                if (r >= 4) {
                    bh0 = bl0;
                    bh1 = bl1;
                }
            }
            pv_page<VB, NT>(tile, tl.off_vc, lane, bh0, bh1, bl0, bl1, oacc, lut);
        }

        // hand the unit's slots back: issue the unit n_grp ahead into them
        __syncwarp();
        if (u + n_grp < n_units) {  // warp-uniform
            fence_proxy_async_smem();
            issue_unit(u + n_grp, st, pid_next);
            n_issued = u + n_grp + 1;
            const int j = BG_UNIT * (u + n_grp + 1) + lane;
            if (lane < BG_UNIT && j < my_count) pid_next = __ldg(bt + page_of(j));
        }
        parity ^= st + 1 == n_grp ? 1u : 0u;
        st = st + 1 == n_grp ? 0 : st + 1;
    }
    if (u_fail >= 0 && lane == 0)
        for (int v = u_fail; v < n_issued; ++v)
            (void)mbar_wait_bounded(&sm.bar[warp][v % n_grp], (v / n_grp) & 1, 1000000LL);
    griddep_launch_dependents();

    // ---- warp partial: normalisers summed over the lanes of each head
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], 4);
        lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], 8);
        lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], 16);
    }
    __syncthreads();  // every warp is done with its ring (o_part takes its place)
    if constexpr (NT == 1) {
        // columns 4..7 (lanes t = 2, 3) hold the low parts of heads 0..3
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[m][e] += __shfl_xor_sync(0xffffffffu, oacc[m][e], 2);
    }
    if (NT == 2 || t < 2) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int c0 = 16 * r + 2 * m;
            if (2 * t < G) {
                o_part[warp][2 * t][c0] = oacc[m][0];
                o_part[warp][2 * t][c0 + 1] = oacc[m][2];
            }
            if (2 * t + 1 < G) {
                o_part[warp][2 * t + 1][c0] = oacc[m][1];
                o_part[warp][2 * t + 1][c0 + 1] = oacc[m][3];
            }
        }
    }
    if (lane < 4) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int jj = 4 * nt + lane;
            if (jj < G) {
                sm.ms.m_part[warp][jj] = mrun[nt];
                sm.ms.l_part[warp][jj] = lsum[nt];
            }
        }
    }
    __syncthreads();
    finish_decode<NW, MAXG>(sm.ms, o_part, G, H_q, H_kv, B, b, h, split, S, ws, pi_table + __ldg(pi_offsets + D),
                            out);
}

}  // namespace kvq

using namespace kvq;

namespace {
// instances by (head group up to 4 / up to 8, value width 1..8)
using BgKernel = decltype(&bgtq_decode_kernel<4, 1>);
const BgKernel kBgKernels[2][8] = {
    {bgtq_decode_kernel<4, 1>, bgtq_decode_kernel<4, 2>, bgtq_decode_kernel<4, 3>, bgtq_decode_kernel<4, 4>,
     bgtq_decode_kernel<4, 5>, bgtq_decode_kernel<4, 6>, bgtq_decode_kernel<4, 7>, bgtq_decode_kernel<4, 8>},
    {bgtq_decode_kernel<8, 1>, bgtq_decode_kernel<8, 2>, bgtq_decode_kernel<8, 3>, bgtq_decode_kernel<8, 4>,
     bgtq_decode_kernel<8, 5>, bgtq_decode_kernel<8, 6>, bgtq_decode_kernel<8, 7>, bgtq_decode_kernel<8, 8>}};

// Dynamic shared memory a kernel may take next to its static tables, opted
// in once per device and kernel.
kvq_status bgtq_dynamic_smem_limit(BgKernel kern, int kid, size_t* limit) {
    static std::mutex mu;
    static size_t lim[64][16] = {};
    int dev = 0;
    kvq_status s = kvq_check_cuda(cudaGetDevice(&dev), "bgtq_decode_attn: cudaGetDevice");
    if (s != KVQ_OK) return s;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && lim[dev][kid]) {
        *limit = lim[dev][kid];
        return KVQ_OK;
    }
    int optin = 0;
    s = kvq_check_cuda(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                       "bgtq_decode_attn: shared-memory limit");
    if (s != KVQ_OK) return s;
    cudaFuncAttributes fa;
    s = kvq_check_cuda(cudaFuncGetAttributes(&fa, (const void*)kern), "bgtq_decode_attn: kernel attributes");
    if (s != KVQ_OK) return s;
    if ((size_t)optin <= fa.sharedSizeBytes)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: no shared memory left next to the tables");
    const size_t dyn = (size_t)optin - fa.sharedSizeBytes;
    s = kvq_check_cuda(cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn),
                       "bgtq_decode_attn smem attribute");
    if (s != KVQ_OK) return s;
    if (dev >= 0 && dev < 64) lim[dev][kid] = dyn;
    *limit = dyn;
    return KVQ_OK;
}
}  // namespace

// one CTA per SM, as the INT2 decode (kvq_decode_auto_splits)
int bgtq_decode_auto_splits(int B, int H_q, int H_kv, int max_pages_per_seq) {
    return kvq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
}

extern "C" kvq_status bgtq_decode_attn(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                       int64_t num_pages, const int32_t* block_table, int max_pages_per_seq,
                                       const int32_t* context_lens, const int8_t* widths, int total_bits, int v_bits,
                                       const float* pi_table, const int64_t* pi_offsets, const double* codebooks,
                                       float scale, float* out, void* workspace, size_t workspace_bytes,
                                       int num_splits, void* stream) {
    kvq_status st = bgtq_check_common("bgtq_decode_attn", d, H_kv, total_bits, v_bits, pi_table);
    if (st != KVQ_OK) return st;
    if (B <= 0 || B > 65535 || H_q <= 0 || H_q % H_kv || max_pages_per_seq <= 0 || num_pages <= 0 || num_splits < 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: B=%d H_q=%d H_kv=%d max_pages=%d", B, H_q, H_kv,
                             max_pages_per_seq);
    const int G = H_q / H_kv;
    if (G > 8) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: GQA group %d > 8", G);
    if (!q || !cache || !block_table || !context_lens || !widths || !pi_table || !pi_offsets || !codebooks || !out ||
        !workspace)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: null pointer");
    if (reinterpret_cast<uintptr_t>(cache) % 16 || reinterpret_cast<uintptr_t>(workspace) % 16 ||
        reinterpret_cast<uintptr_t>(q) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: q, cache and workspace need 16-byte alignment");
    const int S = num_splits > 0 ? num_splits : bgtq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
    if (S > MAX_SPLITS)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: num_splits=%d above %d", S, MAX_SPLITS);
    // header, one ticket per (sequence, KV head), B * H_q * S split partials
    const size_t need = WS_HEADER + tickets_bytes(B, H_kv) + (size_t)B * H_q * S * PART_STRIDE * sizeof(float);
    if (workspace_bytes < need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "bgtq_decode_attn: workspace %zu < %zu bytes", workspace_bytes, need);

    const int tile = (int)bgtq_tile_bytes(total_bits, v_bits);
    const bool small = G <= 4;
    const BgKernel kern = kBgKernels[small ? 0 : 1][v_bits - 1];
    size_t dyn_max = 0;
    st = bgtq_dynamic_smem_limit(kern, (small ? 0 : 8) + v_bits - 1, &dyn_max);
    if (st != KVQ_OK) return st;
    const int NW = small ? BgWarps<4>::NW : BgWarps<8>::NW;
    const size_t fixed = align_up(small ? sizeof(BgDecodeSmem<BgWarps<4>::NW, 4>) : sizeof(BgDecodeSmem<BgWarps<8>::NW, 8>),
                                  128);
    int n_stages = dyn_max > fixed ? (int)((dyn_max - fixed) / ((size_t)NW * tile)) : 0;
    n_stages = n_stages > BG_MAX_STAGES ? BG_MAX_STAGES : n_stages;
    n_stages -= n_stages % BG_UNIT;  // whole units of pages
    if (n_stages < BG_UNIT)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: %d-byte tiles leave no room for a unit of stages", tile);
    const size_t ring = (size_t)NW * n_stages * tile, o_bytes = (size_t)NW * (small ? 4 : 8) * D * sizeof(float);
    const size_t smem = fixed + (ring > o_bytes ? ring : o_bytes);
    if (smem > dyn_max)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: %d-byte tiles leave no room", tile);
    static const RsqrtTab rs = [] {
        RsqrtTab t{};
        for (int i = 1; i <= D / 2; ++i) t.v[i] = 1.0 / std::sqrt((double)(2 * i));
        return t;
    }();
    dim3 grid(S, H_kv, B);
    const cudaError_t e =
        launch_pdl(kern, grid, dim3(NW * 32), smem,
                   static_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(q), H_q, H_kv, G,
                   static_cast<const uint8_t*>(cache), num_pages, block_table, max_pages_per_seq, context_lens, widths,
                   total_bits, v_bits, pi_table, pi_offsets, codebooks, scale * 1.4426950408889634f, out,
                   static_cast<uint8_t*>(workspace), n_stages, rs);
    return kvq_check_cuda(e, "bgtq_decode_attn launch");
}
