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
// of bulk async copies, as in the INT2 decode, three pages per mbarrier
// phase (one wait, one release, one softmax rescale, and one pass over the
// chunk descriptors and B fragments per unit).  Per page (16 tokens):
//   QK  mma.sync m16n8k16 over chunks of 16 gathered positions of one width
//       (a width group padded to a multiple of 16; groups are laid out in
//       ascending width).  Rows = tokens r, r + 8; lane t holds the chunk's
//       RoPE blocks 2t, 2t + 1, whose 4b code bits are contiguous in a
//       token's stream and come out of one 32-bit window.  A = C_b[code] /
//       sqrt(n_b) as an fp16 hi/lo pair from a shared-memory table; B =
//       q~ sigma (a per-head power of two) as hi/lo columns, zero past the
//       group; the token's group norm r_{s,b} scales each chunk's dot
//       products in fp32.
//   softmax  online, base 2, exact running maximum per head; p is rounded to
//       fp16 once (p^), and the same p^ weights the values and the
//       normaliser.
//   PV  mma.sync m16n8k16 with rows = channels, K = the 16 tokens.  Lane
//       (r, t) owns channels 16r .. 16r+15 (one contiguous 16 v_bits-bit
//       field of each token's value stream): the MMA row pair (r, r + 8) of
//       chunk m is channels 16r + 2m, 16r + 2m + 1.  A = C_v[code] / sqrt(128)
//       as fp16 from a shared-memory table; B = p^ r_v as an exact fp16
//       hi/lo pair (HMUL2, then HFMA2 for the remainder) in the N columns.
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
    int bit0;      // first code bit of the chunk in a token's key stream
    int8_t b;      // width
    int8_t last;   // the last chunk of its width group
    int16_t pos0;  // first gathered position
};

template <int NW, int MAXG>
struct __align__(16) BgDecodeSmem {
    uint2 bfr[BG_MAX_CHUNKS][MAXG / 4][32];  // QK B fragments per chunk, n-tile and lane
    uint32_t cbk2[8][256];  // C_b / sqrt(n_b) per width as (fp16 hi | fp16 lo << 16)
    BgChunk chunks[BG_MAX_CHUNKS];
    int n_chunks;
    float sigma[MAXG];      // power-of-two pre-scale per head
    __half pbh[NW][MAXG][BG_UNIT * PAGE];  // p^ of the warp's current unit, head-major
    __half cb_vh[256];         // C_v / sqrt(128) as fp16 (PV A operand)
    float qt[MAXG][D];         // q~ in gathered order, times scale * log2(e)
    float qin[MAXG][D];
    float cb_v[256];           // C_v / sqrt(128)
    uint64_t bar[NW][BG_MAX_STAGES];
    int ntok[NW][BG_MAX_STAGES];
    BgtqLayout L;
    int8_t wsm[D / 2];      // this head's block widths
    MergeSmem<NW, MAXG> ms;
};


template <int MAXG, int VB>
__global__ void __launch_bounds__(BgWarps<MAXG>::NW * 32, 1)
bgtq_decode_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int G, const uint8_t* __restrict__ cache,
                   int64_t num_pages, const int32_t* __restrict__ block_table, int max_pages,
                   const int32_t* __restrict__ context_lens, const int8_t* __restrict__ widths, int total_bits,
                   int v_bits, const float* __restrict__ pi_table, const int64_t* __restrict__ pi_offsets,
                   const double* __restrict__ codebooks, float scale_log2, float* __restrict__ out,
                   uint8_t* __restrict__ ws, int n_stages) {
    constexpr int NW = BgWarps<MAXG>::NW;
    extern __shared__ __align__(128) uint8_t smem_raw[];
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
    int ctx = __ldg(context_lens + b);
    ctx = max(0, min(ctx, max_pages * PAGE));
    const int n_pages = (ctx + PAGE - 1) / PAGE;
    const int32_t* bt = block_table + (size_t)b * max_pages;
    // pages dealt round-robin over all S * NW warps of the (sequence, KV head)
    const int KS = S * NW, k0 = split * NW + warp;
    const int my_count = n_pages > k0 ? (n_pages - k0 + KS - 1) / KS : 0;
    auto page_of = [&](int j) { return k0 + KS * j; };

    // Pages travel in units of BG_UNIT (one mbarrier phase, one wait, one
    // release): unit u is the warp's pages 2u, 2u + 1 in ring slots
    // 2 st, 2 st + 1 of slot group st = u % n_grp.
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
    int pid_next = 0, n_issued = 0;
    {
        int pid_first[BG_MAX_STAGES / BG_UNIT];
#pragma unroll
        for (int u = 0; u < BG_MAX_STAGES / BG_UNIT; ++u) pid_first[u] = 0;
        if (lane < BG_UNIT) {
#pragma unroll
            for (int u = 0; u <= BG_MAX_STAGES / BG_UNIT; ++u) {
                const int j = BG_UNIT * u + lane;
                const int pid = u <= n_grp && j < my_count ? __ldg(bt + page_of(j)) : 0;
                if (u < BG_MAX_STAGES / BG_UNIT) pid_first[u] = pid;
                if (u == n_grp) pid_next = pid;
            }
        }
#pragma unroll
        for (int u = 0; u < BG_MAX_STAGES / BG_UNIT; ++u)
            if (u < n_grp && u < n_units) {  // warp-uniform
                issue_unit(u, u, pid_first[u]);
                n_issued = u + 1;
            }
    }
    {
        // the block table and the output rotation are read later: have L2 keep them
        const char* btc = reinterpret_cast<const char*>(bt);
        const int lines = (n_pages * 4 + 127) / 128;
        for (int l = split * NW * 32 + tid; l < lines; l += S * NW * 32) prefetch_l2_keep(btc + 128 * l);
        const char* rot = reinterpret_cast<const char*>(pi_table + __ldg(pi_offsets + D));
        for (int l = tid; l < D * D * 4 / 128; l += NW * 32) prefetch_l2_keep(rot + 128 * l);
    }

    // ---- per-head layout, chunk schedule, codebooks and rotated queries
    build_layout_cta(widths + h * (D / 2), sm.L, sm.wsm);
    if (tid == 0) {
        int nc = 0;
        for (int bb = 1; bb <= 8; ++bb)
            for (int c = 0; c < (sm.L.n[bb] + 15) / 16 && nc < BG_MAX_CHUNKS; ++c) {
                BgChunk ch;
                ch.bit0 = sm.L.bitstart[bb] + 16 * c * bb;
                ch.b = (int8_t)bb;
                ch.last = (int8_t)(16 * (c + 1) >= sm.L.n[bb]);
                ch.pos0 = (int16_t)(sm.L.start[bb] + 16 * c);
                sm.chunks[nc++] = ch;
            }
        sm.n_chunks = nc;
    }
    const __nv_bfloat16* qb = q + ((size_t)b * H_q + (size_t)h * G) * D;
    for (int idx = tid; idx < G * D; idx += NW * 32) sm.qin[idx / D][idx % D] = __bfloat162float(qb[idx]);
    __syncthreads();
    const bool layout_ok = sm.L.ok && sm.L.total_bits <= 2 * total_bits;
    if (!layout_ok && tid == 0) atomicOr(err_word, ERR_BAD_WIDTHS);
    for (int idx = tid; idx < 8 * 256; idx += NW * 32) {
        const int bb = idx / 256 + 1, c = idx % 256;
        if (c < (1 << bb) && sm.L.n[bb] > 0) {
            // the scaled centroid as an fp16 hi/lo pair (about 22 significant bits)
            const float v = scaled_centroid(codebooks, bb, c, sm.L.n[bb]);
            const __half hi = __float2half_rn(v), lo = __float2half_rn(v - __half2float(hi));
            sm.cbk2[bb - 1][c] = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
        }
    }
    for (int c = tid; c < (1 << VB); c += NW * 32) {
        sm.cb_v[c] = scaled_centroid(codebooks, VB, c, D);
        sm.cb_vh[c] = __float2half_rn(sm.cb_v[c]);
    }
    if (tid < D) {
        // q~ at gathered position p = tid: sum_i q[dim(st + i)] Pi_n[i][p - st]
        const int p = tid;
        float acc[MAXG];
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) acc[jj] = 0.f;
        if (layout_ok) {
            const int bb = group_of(sm.L, p);
            const int st = sm.L.start[bb], n = sm.L.n[bb], j = p - st;
            const float* pi = pi_table + __ldg(pi_offsets + n);
#pragma unroll 16
            for (int i = 0; i < n; ++i) {
                const float pv = __ldg(pi + (size_t)i * n + j);
                const int dm = sm.L.dim[st + i];
#pragma unroll
                for (int jj = 0; jj < MAXG; ++jj)
                    if (jj < G) acc[jj] = fmaf(sm.qin[jj][dm], pv, acc[jj]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) sm.qt[jj][p] = jj < G ? acc[jj] * scale_log2 : 0.f;
    }
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

    constexpr int NT = MAXG / 4;  // n-tiles of 8 columns (4 heads x hi/lo)
    constexpr int VPL = NT;
    const int r = lane >> 2, t = lane & 3;
    // ---- QK B fragments: column n = r -> head 4 nt + (r >> 1), part r & 1
    // (hi / lo of q~ sigma); rows k = 2t, 2t+1 (b0) are the chunk positions
    // 4t, 4t+1 and k = 2t+8, 2t+9 (b1) the positions 4t+2, 4t+3, so a lane's
    // two RoPE blocks are adjacent in the code stream; positions past the
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
    __syncthreads();

    // ---- this lane's value field: channels 16r .. 16r+15, the 16 VB bits
    // at bit 16 VB r of a token's value stream, in VW words from vword on
    // (shifted down by vshift = 0 or 16)
    constexpr int VW = (VB + 1) / 2;
    const int vword = (VB * r) >> 1, vshift = 16 * ((VB * r) & 1);

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

        // ---- QK on the tensor cores, one chunk (16 positions of width b) at
        // a time for both pages of the unit: A = C_b[code] / sqrt(n_b) as an
        // fp16 hi/lo pair, rows = tokens r, r + 8, K = the chunk's positions
        // (lane t: blocks 2t, 2t + 1 of the chunk); the group norm r_{s,b}
        // scales each chunk's dot products.
        float lg[BG_UNIT][NT][2];
        {
            float acc[BG_UNIT][NT][2];
#pragma unroll
            for (int e = 0; e < BG_UNIT; ++e)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[e][nt][0] = acc[e][nt][1] = 0.f;
#pragma unroll 2
            for (int k = 0; k < NC; ++k) {
                const BgChunk ch = sm.chunks[k];  // warp-uniform
                const int bw = ch.b;
                // this lane's blocks 2t, 2t+1 of the chunk: 4 bw contiguous bits
                const int off = ch.bit0 + 4 * t * bw, wi = off >> 5, sh = off & 31;
                const uint32_t* cb = sm.cbk2[bw - 1];
                const uint32_t mask = (1u << bw) - 1u;
                uint2 bb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) bb[nt] = sm.bfr[k][nt][lane];
#pragma unroll
                for (int e = 0; e < BG_UNIT; ++e) {
                    const uint32_t* rec0 = reinterpret_cast<const uint32_t*>(tiles[e] + r * tl.kb);
                    const uint32_t* rec8 = reinterpret_cast<const uint32_t*>(tiles[e] + (r + 8) * tl.kb);
                    const uint32_t x0 = __funnelshift_r(rec0[wi], rec0[wi + 1], sh);
                    const uint32_t x8 = __funnelshift_r(rec8[wi], rec8[wi + 1], sh);
                    // A registers: a0 token r block 2t, a1 token r+8 block 2t,
                    // a2 token r block 2t+1, a3 token r+8 block 2t+1
                    uint32_t ah[4], al[4];
                    const uint32_t xs[4] = {x0, x8, x0 >> (2 * bw), x8 >> (2 * bw)};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t e0 = cb[xs[j] & mask], e1 = cb[(xs[j] >> bw) & mask];
                        ah[j] = prmt(e0, e1, 0x5410);
                        al[j] = prmt(e0, e1, 0x7632);
                    }
                    const __half* nrm = reinterpret_cast<const __half*>(tiles[e] + tl.off_kn + 2 * (bw - 1));
                    const float rn0 = __half2float(nrm[8 * r]), rn8 = __half2float(nrm[8 * (r + 8)]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float c[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_f16_16816(c, ah, bb[nt].x, bb[nt].y);
                        mma_f16_16816(c, al, bb[nt].x, bb[nt].y);
                        acc[e][nt][0] = fmaf(rn0, c[0] + c[1], acc[e][nt][0]);
                        acc[e][nt][1] = fmaf(rn8, c[2] + c[3], acc[e][nt][1]);
                    }
                }
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
            const int hq = VPL == 1 ? (r & 3) : r;
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
            if constexpr (VPL == 1) {
                if (r >= 4) {
                    bh0 = bl0;
                    bh1 = bl1;
                }
            }

            // this lane's value fields of tokens 2t, 2t+1, 2t+8, 2t+9, aligned
            uint32_t f[4][VW];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s_tok = 2 * t + (k & 1) + 8 * (k >> 1);
                const uint32_t* vr = reinterpret_cast<const uint32_t*>(tile + tl.off_vc + s_tok * tl.vb) + vword;
                uint32_t w[VW];
#pragma unroll
                for (int q2 = 0; q2 < VW; ++q2) w[q2] = vr[q2];
#pragma unroll
                for (int q2 = 0; q2 < VW; ++q2) f[k][q2] = __funnelshift_r(w[q2], q2 + 1 < VW ? w[q2 + 1] : 0u, vshift);
            }
            // code of channel 16r + i in field k
            auto code = [&](int k, int i) -> uint32_t {
                const int bit = VB * i, wi = bit >> 5, sh = bit & 31;
                uint32_t x = f[k][wi] >> sh;
                if (sh + VB > 32) x |= f[k][wi + 1] << (32 - sh);
                return x & ((1u << VB) - 1u);
            };
            const unsigned short* cbv = reinterpret_cast<const unsigned short*>(sm.cb_vh);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t hv[4][2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    hv[k][0] = cbv[code(k, 2 * m)];
                    hv[k][1] = cbv[code(k, 2 * m + 1)];
                }
                const uint32_t a[4] = {hv[0][0] | (hv[1][0] << 16), hv[0][1] | (hv[1][1] << 16),
                                       hv[2][0] | (hv[3][0] << 16), hv[2][1] | (hv[3][1] << 16)};
                mma_f16_16816(oacc[m], a, bh0, bh1);
                if constexpr (VPL == 2) mma_f16_16816(oacc[m], a, bl0, bl1);
            }
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
    if constexpr (VPL == 1) {
        // columns 4..7 (lanes t = 2, 3) hold the low parts of heads 0..3
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[m][e] += __shfl_xor_sync(0xffffffffu, oacc[m][e], 2);
    }
    if (VPL == 2 || t < 2) {
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
    if (reinterpret_cast<uintptr_t>(cache) % 16 || reinterpret_cast<uintptr_t>(workspace) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: cache and workspace need 16-byte alignment");
    const int S = num_splits > 0 ? num_splits : bgtq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
    if (S > MAX_SPLITS)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_decode_attn: num_splits=%d above %d", S, MAX_SPLITS);
    // header, one ticket per (sequence, KV head), B * H_q * S split partials
    const size_t need = WS_HEADER + tickets_bytes(B, H_kv) + (size_t)B * H_q * S * PART_STRIDE * sizeof(float);
    if (workspace_bytes < need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "bgtq_decode_attn: workspace %zu < %zu bytes", workspace_bytes, need);

    const int tile = (int)bgtq_tile_bytes(total_bits, v_bits);
    constexpr size_t kSmemMax = 227 * 1024;
    const bool small = G <= 4;
    const int NW = small ? BgWarps<4>::NW : BgWarps<8>::NW;
    const size_t fixed = align_up(small ? sizeof(BgDecodeSmem<BgWarps<4>::NW, 4>) : sizeof(BgDecodeSmem<BgWarps<8>::NW, 8>),
                                  128);
    int n_stages = (int)((kSmemMax - fixed) / ((size_t)NW * tile));
    n_stages = n_stages > BG_MAX_STAGES ? BG_MAX_STAGES : n_stages;
    n_stages -= n_stages % BG_UNIT;  // whole units of pages
    if (n_stages < BG_UNIT)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: %d-byte tiles leave no room for a unit of stages", tile);
    const size_t ring = (size_t)NW * n_stages * tile, o_bytes = (size_t)NW * (small ? 4 : 8) * D * sizeof(float);
    const size_t smem = fixed + (ring > o_bytes ? ring : o_bytes);
    if (smem > kSmemMax)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: %d-byte tiles leave no room", tile);
    const BgKernel kern = kBgKernels[small ? 0 : 1][v_bits - 1];
    const int kid = (small ? 0 : 8) + v_bits - 1;
    {
        // opt in once per device and kernel, to the full shared-memory size
        static std::mutex mu;
        static bool done[64][16] = {};
        int dev = 0;
        kvq_status s2 = kvq_check_cuda(cudaGetDevice(&dev), "bgtq_decode_attn: cudaGetDevice");
        if (s2 != KVQ_OK) return s2;
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !done[dev][kid]) {
            s2 = kvq_check_cuda(
                cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax),
                "bgtq_decode_attn smem attribute");
            if (s2 != KVQ_OK) return s2;
            if (dev >= 0 && dev < 64) done[dev][kid] = true;
        }
    }
    dim3 grid(S, H_kv, B);
    const cudaError_t e =
        launch_pdl(kern, grid, dim3(NW * 32), smem,
                   static_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(q), H_q, H_kv, G,
                   static_cast<const uint8_t*>(cache), num_pages, block_table, max_pages_per_seq, context_lens, widths,
                   total_bits, v_bits, pi_table, pi_offsets, codebooks, scale * 1.4426950408889634f, out,
                   static_cast<uint8_t*>(workspace), n_stages);
    return kvq_check_cuda(e, "bgtq_decode_attn launch");
}
