// Fused packed-cache decode attention over the rotated INT2 cache.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization" §3 Eqs. (1)-(2)
// with Eq. (4) folded in: <q, Q2(zR)R^T> = <qR, Q2(zR)>, so the query is
// rotated once (q' = q R_k), the cache is consumed in the rotated basis and
// the output is rotated back once (o = o' R_v^T).  The kernel reads only the
// packed codes and fp16 (scale, min) pairs.
//
// Grid (split, kv_head, seq) with one large CTA per SM (12 warps for head
// groups up to 4, 8 for groups of 8).  Each warp streams pages through its
// own 9-slot ring of 1536-byte tiles filled by bulk async copies
// (cp.async.bulk + mbarrier).  The pages of a (sequence, KV head) are dealt
// round-robin over all warps of its split CTAs.  Per page (16 tokens):
//
//   QK  logit(s, j) = sum_g [ scale_{s,g} <q'_{j,g}, c_{s,g}> + min_{s,g} S_{j,g} ]
//       The 2-bit codes c are fed to mma.sync m16n8k16 as exact fp16
//       subnormals (code << 2k reinterpreted is code * 4^k * 2^-24), one MMA
//       pair per 32-channel group so the group scale applies afterwards; q'
//       enters as an fp16 hi/lo pair (fp16 + fp16 ~ 22 bits) in the eight N
//       columns, pre-scaled by 4^-k and a per-head power of two.
//   softmax  online, base 2, exact running maximum per head.
//   PV  o'(j, i) = sum_s p_{s,j} scale_{s,g} c_{s,i} + sum_s p_{s,j} min_{s,g}
//       rows = channels (codes again as fp16 subnormals), K = the 16 tokens.
//       p is rounded to fp16 once (p^); B = p^ * scale as an exact fp16
//       hi/lo pair (HMUL2, then HFMA2 for the remainder), so the large
//       group minima and the code term cancel without amplifying rounding;
//       the min term is one more MMA with A = the fp16 mins of the groups.
//   Pages travel in units of three (one mbarrier phase, one wait, one
//   release, one softmax rescale per unit); the QK of unit u + 1 and the
//   softmax/PV of unit u are software-pipelined.
//
// Split partials (m, l, o') go to the workspace; the last CTA of a
// (sequence, KV head) to finish (atomic ticket, no waiting) merges them,
// applies R_v^T and writes the output.
#include <mutex>

#include "merge.cuh"

namespace kvq {

constexpr int DEC_STAGES = 9;  // page slots per warp
constexpr int UNIT_PAGES = 3;  // pages per mbarrier phase (one wait, one release)
constexpr int DEC_UNITS = DEC_STAGES / UNIT_PAGES;
static_assert(DEC_STAGES % UNIT_PAGES == 0, "a unit is a whole number of page slots");

// Warps per CTA.  Each of the SM's four schedulers owns a quarter of its
// 64K registers: three warps of 168 registers fit one (head groups up to 4),
// while groups of 8 need more registers per thread and run two per scheduler.
template <int NT>
struct DecWarps {
    static constexpr int NW = NT == 1 ? 12 : 8;
};

template <int NW, int MAXG>
struct __align__(16) DecodeSmem {
    union {
        uint8_t ring[NW][DEC_STAGES][INT2_TILE];  // page tiles in flight
        float o_part[NW][MAXG][D];                // per-warp o' after the loop
    } u;
    uint64_t bar[NW][DEC_UNITS];
    int ntok[NW][DEC_STAGES];  // valid tokens of the page in each stage (0: skipped page)
    float q[MAXG][D];          // scaled rotated queries q~ = q R_k * scale * log2(e)
    float gsum[MAXG][NGROUP];
    float sigma[MAXG];         // power-of-two pre-scale per head
    MergeSmem<NW, MAXG> ms;
};

// BF16 window (the INT2 paper keeps a small BF16 window, §3.1; the
// Block-GTQ page keeps 4 sink and 128 recent tokens, Table 6): the first
// win_lens[b] rows of win_k / win_v [B][win_max][H_kv][d] are attended
// exactly, in the original basis, with the logit q . (k - mu) * scale: the
// same shift by -q . mu that centring gives the cached keys, so the two
// parts share one softmax.  Each warp runs an online softmax over tokens
// warp, warp + NW, ...; lanes hold 4 channels; results go to the per-warp
// partial slots the split finish merges.
template <int NW, int MAXG>
__device__ __forceinline__ void window_partials(float (*o_part)[MAXG][D], MergeSmem<NW, MAXG>& ms,
                                                const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int G, int b,
                                                int h, const float* __restrict__ mu,
                                                const __nv_bfloat16* __restrict__ win_k,
                                                const __nv_bfloat16* __restrict__ win_v,
                                                const int32_t* __restrict__ win_lens, int win_max, float scale_log2) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wl = max(0, min(__ldg(win_lens + b), win_max));
    float qv[MAXG][4], mc[4];
    const __nv_bfloat16* qb = q + ((size_t)b * H_q + (size_t)h * G) * D + 4 * lane;
#pragma unroll
    for (int jj = 0; jj < MAXG; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) qv[jj][e] = jj < G ? __bfloat162float(qb[(size_t)jj * D + e]) : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) mc[e] = __ldg(mu + (size_t)h * D + 4 * lane + e);
    float m_w[MAXG], l_w[MAXG], o_w[MAXG][4];
#pragma unroll
    for (int jj = 0; jj < MAXG; ++jj) {
        m_w[jj] = -CUDART_INF_F;
        l_w[jj] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) o_w[jj][e] = 0.f;
    }
    for (int t = warp; t < wl; t += NW) {
        const size_t row = (((size_t)b * win_max + t) * H_kv + h) * D + 4 * lane;
        const uint2 kr = __ldg(reinterpret_cast<const uint2*>(win_k + row));
        const uint2 vr = __ldg(reinterpret_cast<const uint2*>(win_v + row));
        const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kr.x));
        const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kr.y));
        const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr.x));
        const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr.y));
        const float kc[4] = {__fsub_rn(k01.x, mc[0]), __fsub_rn(k01.y, mc[1]), __fsub_rn(k23.x, mc[2]),
                             __fsub_rn(k23.y, mc[3])};
        const float vc[4] = {v01.x, v01.y, v23.x, v23.y};
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) {
            if (jj >= G) continue;
            float dot = qv[jj][0] * kc[0];
#pragma unroll
            for (int e = 1; e < 4; ++e) dot = fmaf(qv[jj][e], kc[e], dot);
#pragma unroll
            for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const float lg = dot * scale_log2;
            const float mn = fmaxf(m_w[jj], lg);
            const float corr = ex2(m_w[jj] - mn);  // 0 while nothing was seen
            const float p = ex2(lg - mn);
            l_w[jj] = fmaf(l_w[jj], corr, p);
#pragma unroll
            for (int e = 0; e < 4; ++e) o_w[jj][e] = fmaf(o_w[jj][e], corr, p * vc[e]);
            m_w[jj] = mn;
        }
    }
#pragma unroll
    for (int jj = 0; jj < MAXG; ++jj)
        if (jj < G) {
#pragma unroll
            for (int e = 0; e < 4; ++e) o_part[warp][jj][4 * lane + e] = o_w[jj][e];
            if (lane == 0) {
                ms.m_part[warp][jj] = m_w[jj];
                ms.l_part[warp][jj] = l_w[jj];
            }
        }
}

// WIN: the grid's last split attends the BF16 window (a separate
// instantiation, so the plain decode carries none of it).
template <int NT, bool WIN>
__global__ void __launch_bounds__(DecWarps<NT>::NW * 32, 1)
decode_int2_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int G, const uint8_t* __restrict__ cache,
                   int64_t num_pages, const int32_t* __restrict__ block_table, int max_pages,
                   const int32_t* __restrict__ context_lens, const float* __restrict__ Rk,
                   const float* __restrict__ Rv, const float* __restrict__ mu,
                   const __nv_bfloat16* __restrict__ win_k, const __nv_bfloat16* __restrict__ win_v,
                   const int32_t* __restrict__ win_lens, int win_max, float scale_log2, float* __restrict__ out,
                   uint8_t* __restrict__ ws) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int MAXG = 4 * NT;
    constexpr int NW = DecWarps<NT>::NW;
    DecodeSmem<NW, MAXG>& sm = *reinterpret_cast<DecodeSmem<NW, MAXG>*>(smem_raw);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int S = gridDim.x, B = gridDim.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, t = lane & 3;

    uint32_t* err_word = reinterpret_cast<uint32_t*>(ws);

    // The rotations are constants of the layer: this warp's rows of R_k are
    // loaded, and R_v (read only after the loop) fetched into L2, while the
    // previous kernel in the stream may still be running.
    float4 rr[RowPrefetch<NW, MAXG>::N];
    load_rows<NW>(Rk + (size_t)h * D * D, rr);
    {
        const char* rv = reinterpret_cast<const char*>(Rv + (size_t)h * D * D);
        for (int l = tid; l < D * D * 4 / 128; l += NW * 32) prefetch_l2_keep(rv + 128 * l);
    }
    {
        // The inputs the prologue reads first -- this warp's first block-table
        // entries, the context length, the query rows -- are only prefetched
        // into L2 here; the loads that use them follow the wait.
        const int S_pf = WIN ? S - 1 : S, k0_pf = split * NW + warp;
        const int j = k0_pf + S_pf * NW * lane;
        if (lane < DEC_STAGES + UNIT_PAGES && j < max_pages) prefetch_l2(block_table + (size_t)b * max_pages + j);
        if (tid == 0) prefetch_l2(context_lens + b);
        const char* qc = reinterpret_cast<const char*>(q + ((size_t)b * H_q + (size_t)h * G) * D);
        if (tid < (G * D * 2 + 127) / 128) prefetch_l2(qc + 128 * tid);
    }
    griddep_wait();  // every other input may come from the previous kernel in the stream
    if constexpr (WIN) {
        if (split == S - 1) {
            // the last split attends the BF16 window instead of cache pages
            griddep_launch_dependents();
            window_partials<NW, MAXG>(sm.u.o_part, sm.ms, q, H_q, H_kv, G, b, h, mu, win_k, win_v, win_lens, win_max,
                                      scale_log2);
            __syncthreads();
            finish_decode<NW, MAXG, false>(sm.ms, sm.u.o_part, G, H_q, H_kv, B, b, h, split, S, ws, nullptr, out);
            return;
        }
    }
    const int S_pages = WIN ? S - 1 : S;  // splits that stream cache pages
    int ctx = __ldg(context_lens + b);
    ctx = max(0, min(ctx, max_pages * PAGE));
    const int n_pages = (ctx + PAGE - 1) / PAGE;
    const int32_t* bt = block_table + (size_t)b * max_pages;
    // Page schedule: the pages of a (sequence, KV head) are dealt round-robin
    // over all S * NW warps of its split CTAs, so warp k0 = split * NW + warp
    // takes pages k0, k0 + KS, k0 + 2 KS, ...  Every warp gets the same
    // number of pages to within one, and page ids come from anywhere in the
    // sequence (the block table scatters them over the cache anyway).
    const int KS = S_pages * NW, k0 = split * NW + warp;
    const int my_count = n_pages > k0 ? (n_pages - k0 + KS - 1) / KS : 0;
    auto page_of = [&](int j) { return k0 + KS * j; };

    constexpr int QPT = (MAXG * D + NW * 32 - 1) / (NW * 32);  // query values per thread
    // the query loads go out before lane 0 waits for its page ids, so the
    // two global round trips overlap
    float qv[QPT];
    {
        const __nv_bfloat16* qb = q + ((size_t)b * H_q + (size_t)h * G) * D;
#pragma unroll
        for (int k = 0; k < QPT; ++k) {
            const int idx = tid + k * NW * 32;
            qv[k] = idx < G * D ? __bfloat162float(qb[idx]) : 0.f;
        }
    }
    // Pages travel in units of UNIT_PAGES: unit u holds the warp's pages
    // UNIT_PAGES u .. UNIT_PAGES u + UNIT_PAGES - 1 (ring slots j % DEC_STAGES) on
    // one mbarrier phase, so a unit costs one wait and one release.
    const int n_units = (my_count + UNIT_PAGES - 1) / UNIT_PAGES;
    if (lane == 0) {
        for (int s = 0; s < DEC_UNITS; ++s) mbar_init(&sm.bar[warp][s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    // Lane 0 issues unit u with its (already loaded) page ids and records how
    // many tokens of each page are valid (0 for a slot past the warp's pages
    // or with a bad page id); the mbarrier publishes the counts with the data.
    auto issue_unit = [&](int u, int st, int pid) {
        // whole warp; lane e < UNIT_PAGES issues page e of unit u (id pid),
        // st = u % DEC_UNITS
        uint64_t* bar = &sm.bar[warp][st];
        const int j = UNIT_PAGES * u + lane;
        bool ok = false;
        if (lane < UNIT_PAGES) {
            int n = 0;
            if (j < my_count) {
                if (pid < 0 || (int64_t)pid >= num_pages) {
                    atomicOr(err_word, ERR_BAD_PAGE);
                } else {
                    ok = true;
                    n = min(PAGE, ctx - page_of(j) * PAGE);
                }
            }
            sm.ntok[warp][UNIT_PAGES * st + lane] = n;
        }
        const uint32_t n_ok = __popc(__ballot_sync(0xffffffffu, ok));
        __syncwarp();  // the lanes' counts are ordered before lane 0's arrive (release)
        if (lane == 0) {
            if (n_ok == 0)
                mbar_arrive(bar);  // complete the phase without data
            else
                mbar_arrive_expect_tx(bar, n_ok * INT2_TILE);
        }
        __syncwarp();  // the expected bytes are set before any copy is issued
        if (ok)
            bulk_g2s(sm.u.ring[warp][UNIT_PAGES * st + lane], cache + ((size_t)pid * H_kv + h) * INT2_TILE,
                     INT2_TILE, bar);
    };
    // ---- the page ids of the first units (lane e < UNIT_PAGES holds page e
    // of each).  Their copies are issued after the query rotation, which runs
    // while the ids arrive; the copies then fly during the B-fragment setup.
    // Lanes keep the ids of the next unit to issue, loaded one release
    // before their use.
    int pid_first[DEC_UNITS];
    int pid_next = 0;
    int n_issued = 0;  // units issued so far
#pragma unroll
    for (int u = 0; u < DEC_UNITS; ++u) pid_first[u] = 0;
    if (lane < UNIT_PAGES) {
        // bounded by the block table's row length, not the context, so these
        // loads need not wait for context_lens
#pragma unroll
        for (int u = 0; u <= DEC_UNITS; ++u) {
            const int j = page_of(UNIT_PAGES * u + lane);
            const int pid = j < max_pages ? __ldg(bt + j) : 0;
            if (u < DEC_UNITS)
                pid_first[u] = pid;
            else
                pid_next = pid;
        }
    }

    // ---- q~ = (q R_k) * scale * log2(e) for the G heads of this KV head
    {
#pragma unroll
        for (int k = 0; k < QPT; ++k) {
            const int idx = tid + k * NW * 32;
            if (idx < G * D) sm.ms.o_final[idx / D][idx % D] = qv[k];
        }
        __syncthreads();
        rotate_rows<NW, MAXG>(sm.ms.o_final, Rk + (size_t)h * D * D, rr, G, scale_log2, sm.q, sm.ms);
#pragma unroll
        for (int u = 0; u < DEC_UNITS; ++u)
            if (u < n_units) {  // warp-uniform
                issue_unit(u, u, pid_first[u]);
                n_issued = u + 1;
            }
        {
            // the rest of this sequence's block table is read one entry at a
            // time during the loop: have L2 fetch it now (after the rotation,
            // which need not wait for the context length this bound needs)
            const char* btc = reinterpret_cast<const char*>(bt);
            const int lines = (n_pages * 4 + 127) / 128;
            for (int l = split * NW * 32 + tid; l < lines; l += S_pages * NW * 32) prefetch_l2_keep(btc + 128 * l);
        }
        // per head: power-of-two pre-scale (max |q~| * sigma in [2^14, 2^15)) and group sums
        for (int jj = warp; jj < G; jj += NW) {
            float mx = 0.f;
            float gs[NGROUP];
#pragma unroll
            for (int g = 0; g < NGROUP; ++g) {
                const float x = sm.q[jj][32 * g + lane];
                mx = fmaxf(mx, fabsf(x));
                gs[g] = x;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
                for (int g = 0; g < NGROUP; ++g) gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], o);
            }
            if (lane == 0) {
                sm.sigma[jj] = mx > 0.f ? ldexpf(1.f, 14 - ilogbf(mx)) : 1.f;
#pragma unroll
                for (int g = 0; g < NGROUP; ++g) sm.gsum[jj][g] = gs[g];
            }
        }
        __syncthreads();
    }

    // ---- QK B fragments: column n = r -> head 4*nt + (r >> 1), part r & 1 (hi / lo)
    uint32_t bq[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hq = 4 * nt + (r >> 1);
        const bool lo_part = r & 1;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int g = s >> 1, hs = s & 1;
#pragma unroll
            for (int e = 0; e < 2; ++e) {  // b0 (k = 2hs), b1 (k = 2hs + 1)
                const int k = 2 * hs + e;
                const int c0 = 32 * g + 8 * t + k, c1 = c0 + 4;
                float v0 = 0.f, v1 = 0.f;
                if (hq < G) {
                    const float f = sm.sigma[hq] * (k == 0 ? 1.f : k == 1 ? 0.25f : k == 2 ? 0.0625f : 0.015625f);
                    v0 = sm.q[hq][c0] * f;
                    v1 = sm.q[hq][c1] * f;
                }
                // hi part (even columns) or the exact remainder (odd columns), one path
                const float h0 = __half2float(__float2half_rn(v0)), h1 = __half2float(__float2half_rn(v1));
                bq[nt][s][e] = pack_half2(lo_part ? v0 - h0 : h0, lo_part ? v1 - h1 : h1);
            }
        }
    }
    float inv_sig[NT], gsum[NT][NGROUP];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hq = 4 * nt + t;
        inv_sig[nt] = hq < G ? 16777216.f / sm.sigma[hq] : 0.f;
#pragma unroll
        for (int g = 0; g < NGROUP; ++g) gsum[nt][g] = hq < G ? sm.gsum[hq][g] : 0.f;
    }

    float oacc[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[m][e] = 0.f;
    float cmin[4] = {0.f, 0.f, 0.f, 0.f};
    float mrun[NT], lsum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrun[nt] = -CUDART_INF_F;
        lsum[nt] = 0.f;
    }

    // Wait for unit u of this warp; false on a timeout.  On a sequence's
    // last page the slots past the context may hold stale bytes (even NaN
    // scales), and so does a slot with no page: their value scale/min words
    // are zeroed here, so p = 0
    // always meets finite factors and the PV step needs no per-slot masks
    // (the QK step drops those slots' logits by selection).
    auto wait_unit = [&](int st, uint32_t parity) -> bool {  // slot group st = u % DEC_UNITS
        const bool ok = mbar_wait_bounded(&sm.bar[warp][st], parity, WAIT_LIMIT_CYCLES);
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) atomicOr(err_word, ERR_TIMEOUT);
            return false;
        }
        bool short_page = false;
#pragma unroll
        for (int e = 0; e < UNIT_PAGES; ++e) short_page |= sm.ntok[warp][UNIT_PAGES * st + e] < PAGE;
        if (short_page) {  // warp-uniform
            // 64 meta words per page (32 scale, 32 min words of slot pairs):
            // clear the halves of slots at or past the page's token count
            for (int k = lane; k < UNIT_PAGES * 64; k += 32) {
                const int e = k >> 6, w = k & 63, pair = (w & 31) >> 2;
                const int n = sm.ntok[warp][UNIT_PAGES * st + e];
                const uint32_t keep = (2 * pair < n ? 0x0000ffffu : 0u) | (2 * pair + 1 < n ? 0xffff0000u : 0u);
                uint32_t* word = reinterpret_cast<uint32_t*>(sm.u.ring[warp][UNIT_PAGES * st + e] + OFF_VM) + w;
                if (keep != 0xffffffffu) *word &= keep;
            }
            __syncwarp();
        }
        return true;
    };

    // ---------------- QK of the page in ring slot `slot`: base-2 logits of tokens r, r + 8 for
    // head 4*nt + t (-inf past the context)
    auto qk_page = [&](int slot, float (&lg)[NT][2]) {
        const uint8_t* tile = sm.u.ring[warp][slot];
        const int n_tok = sm.ntok[warp][slot];
        const uint2 kr = lds64(tile + OFF_KC + 32 * r + 8 * t);
        const uint2 kr8 = lds64(tile + OFF_KC + 32 * (r + 8) + 8 * t);
        const uint32_t P01 = prmt(kr.x, kr.y, 0x5410), P23 = prmt(kr.x, kr.y, 0x7632);
        const uint32_t Q01 = prmt(kr8.x, kr8.y, 0x5410), Q23 = prmt(kr8.x, kr8.y, 0x7632);
        const uint4 mr = lds128(tile + OFF_KM + 16 * r);
        const uint4 mr8 = lds128(tile + OFF_KM + 16 * (r + 8));
        const uint32_t mrw[4] = {mr.x, mr.y, mr.z, mr.w}, mr8w[4] = {mr8.x, mr8.y, mr8.z, mr8.w};
        float acc_r[NT], acc_r8[NT], mn_r[NT], mn_r8[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc_r[nt] = acc_r8[nt] = mn_r[nt] = mn_r8[nt] = 0.f;
#pragma unroll
        for (int g = 0; g < NGROUP; ++g) {
            const uint32_t xr = g == 0 ? P01 : g == 1 ? (P01 >> 8) : g == 2 ? P23 : (P23 >> 8);
            const uint32_t xr8 = g == 0 ? Q01 : g == 1 ? (Q01 >> 8) : g == 2 ? Q23 : (Q23 >> 8);
            const float2 smr = __half22float2(u32_as_h2(mrw[g]));    // (scale, min) token r
            const float2 smr8 = __half22float2(u32_as_h2(mr8w[g]));  // token r + 8
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hs = 0; hs < 2; ++hs) {
                    const uint32_t m0 = 0x00030003u << (4 * hs), m1 = 0x00030003u << (4 * hs + 2);
                    const uint32_t a[4] = {xr & m0, xr8 & m0, xr & m1, xr8 & m1};
                    mma_f16_16816(c, a, bq[nt][2 * g + hs][0], bq[nt][2 * g + hs][1]);
                }
                acc_r[nt] = fmaf(smr.x, c[0] + c[1], acc_r[nt]);
                acc_r8[nt] = fmaf(smr8.x, c[2] + c[3], acc_r8[nt]);
                mn_r[nt] = fmaf(smr.y, gsum[nt][g], mn_r[nt]);
                mn_r8[nt] = fmaf(smr8.y, gsum[nt][g], mn_r8[nt]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            lg[nt][0] = r < n_tok ? fmaf(acc_r[nt], inv_sig[nt], mn_r[nt]) : -CUDART_INF_F;
            lg[nt][1] = r + 8 < n_tok ? fmaf(acc_r8[nt], inv_sig[nt], mn_r8[nt]) : -CUDART_INF_F;
        }
    };

    // QK of unit u and each head's maximum over its pages
    auto qk_unit = [&](int st, float (&lg)[UNIT_PAGES][NT][2], float (&pm)[NT]) {
#pragma unroll
        for (int e = 0; e < UNIT_PAGES; ++e) qk_page(UNIT_PAGES * st + e, lg[e]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float m = fmaxf(lg[0][nt][0], lg[0][nt][1]);
#pragma unroll
            for (int e = 1; e < UNIT_PAGES; ++e) m = fmaxf(m, fmaxf(lg[e][nt][0], lg[e][nt][1]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            pm[nt] = m;
        }
    };

    // ---------------- online softmax (base 2) for one unit, head 4*nt + t:
    // raise the running maxima, rescale the accumulators when one grew, and
    // return p^ (p rounded to fp16 once; the same p^ weights the codes, the
    // group minima and the normaliser)
    auto softmax_unit = [&](const float (&lg)[UNIT_PAGES][NT][2], const float (&pm)[NT], float (&pr)[UNIT_PAGES][NT][2]) {
        float corr[NT];
        bool need = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            corr[nt] = 1.f;
            if (pm[nt] > mrun[nt]) {
                corr[nt] = ex2(mrun[nt] - pm[nt]);  // 0 when mrun = -inf
                mrun[nt] = pm[nt];
                need = true;
            }
            const float mref = mrun[nt] == -CUDART_INF_F ? 0.f : mrun[nt];
#pragma unroll
            for (int e = 0; e < UNIT_PAGES; ++e) {
                pr[e][nt][0] = __half2float(__float2half_rn(ex2(lg[e][nt][0] - mref)));
                pr[e][nt][1] = __half2float(__float2half_rn(ex2(lg[e][nt][1] - mref)));
            }
            float ps = pr[0][nt][0] + pr[0][nt][1];
#pragma unroll
            for (int e = 1; e < UNIT_PAGES; ++e) ps += pr[e][nt][0] + pr[e][nt][1];
            lsum[nt] = fmaf(lsum[nt], corr[nt], ps);
        }
        if (__any_sync(0xffffffffu, need)) {
            // PV columns 2t, 2t+1 hold heads 2t, 2t+1, whose maxima live in lanes (2t)&3, (2t+1)&3
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
            cmin[0] *= cA;
            cmin[2] *= cA;
            cmin[1] *= cB;
            cmin[3] *= cB;
        }
    };

    // ---------------- PV of the page in ring slot `slot` with its weights p^
    auto pv_page = [&](int slot, const float (&pr)[NT][2]) {
        const uint8_t* tile = sm.u.ring[warp][slot];
        // P in the PV B layout: column n = r (head n), rows = tokens 2t, 2t+1 | 2t+8, 2t+9
        uint32_t pb0, pb1;
        {
            const uint32_t X0 = pack_half2(pr[0][0], pr[0][1]);  // (token r, token r+8) of head t
            const int srcA = 8 * t + (r & 3), srcB = 8 * t + 4 + (r & 3);
            uint32_t Y0 = __shfl_sync(0xffffffffu, X0, srcA), Y1 = __shfl_sync(0xffffffffu, X0, srcB);
            if constexpr (NT == 2) {
                const uint32_t X1 = pack_half2(pr[1][0], pr[1][1]);
                const uint32_t Z0 = __shfl_sync(0xffffffffu, X1, srcA), Z1 = __shfl_sync(0xffffffffu, X1, srcB);
                if (r >= 4) {
                    Y0 = Z0;
                    Y1 = Z1;
                }
            }
            // NT == 1: columns 4..7 repeat heads 0..3 and carry the low part of p*scale
            if ((NT == 1 ? (r & 3) : r) >= G) Y0 = Y1 = 0u;
            pb0 = prmt(Y0, Y1, 0x5410);  // p(2t), p(2t+1)
            pb1 = prmt(Y0, Y1, 0x7632);  // p(2t+8), p(2t+9)
        }
        // value scales of tokens (2t, 2t+1) and (2t+8, 2t+9), one word per group
        const uint4 sA = lds128(tile + OFF_VM + 16 * t);
        const uint4 sB = lds128(tile + OFF_VM + 16 * (t + 4));
        const uint32_t wA[4] = {sA.x, sA.y, sA.z, sA.w}, wB[4] = {sB.x, sB.y, sB.z, sB.w};

        // min term: rows = groups (rows 4..15 are never read), K = tokens
        {
            uint32_t a[4] = {0u, 0u, 0u, 0u};
            a[0] = lds32(tile + OFF_VM + VM_MINS + 16 * t + 4 * (r & 3));
            a[2] = lds32(tile + OFF_VM + VM_MINS + 16 * (t + 4) + 4 * (r & 3));
            mma_f16_16816(cmin, a, pb0, pb1);
        }

        const uint32_t v0 = lds32(tile + OFF_VC + 32 * (2 * t) + 4 * r);
        const uint32_t v1 = lds32(tile + OFF_VC + 32 * (2 * t + 1) + 4 * r);
        const uint32_t v8 = lds32(tile + OFF_VC + 32 * (2 * t + 8) + 4 * r);
        const uint32_t v9 = lds32(tile + OFF_VC + 32 * (2 * t + 9) + 4 * r);
        const uint32_t A01 = prmt(v0, v1, 0x5410), A23 = prmt(v0, v1, 0x7632);
        const uint32_t B01 = prmt(v8, v9, 0x5410), B23 = prmt(v8, v9, 0x7632);
        const __half2 P0 = u32_as_h2(pb0), P1 = u32_as_h2(pb1);
#pragma unroll
        for (int g = 0; g < NGROUP; ++g) {
            const uint32_t xa = g == 0 ? A01 : g == 1 ? (A01 >> 8) : g == 2 ? A23 : (A23 >> 8);
            const uint32_t xb = g == 0 ? B01 : g == 1 ? (B01 >> 8) : g == 2 ? B23 : (B23 >> 8);
            // p^ * scale exactly as an fp16 pair: hi = rn(p^ s), lo = p^ s - hi (exact)
            const __half2 S01 = u32_as_h2(wA[g]), S89 = u32_as_h2(wB[g]);
            const __half2 H0 = __hmul2(P0, S01), H1 = __hmul2(P1, S89);
            const __half2 L0 = __hfma2(P0, S01, __hneg2(H0)), L1 = __hfma2(P1, S89, __hneg2(H1));
#pragma unroll
            for (int hs = 0; hs < 2; ++hs) {
                const uint32_t k0 = 0x00030003u << (4 * hs), k1 = 0x00030003u << (4 * hs + 2);
                const uint32_t a[4] = {xa & k0, xa & k1, xb & k0, xb & k1};
                if constexpr (NT == 1) {
                    const bool lo = r >= 4;
                    mma_f16_16816(oacc[2 * g + hs], a, h2_as_u32(lo ? L0 : H0), h2_as_u32(lo ? L1 : H1));
                } else {
                    mma_f16_16816(oacc[2 * g + hs], a, h2_as_u32(H0), h2_as_u32(H1));
                    mma_f16_16816(oacc[2 * g + hs], a, h2_as_u32(L0), h2_as_u32(L1));
                }
            }
        }
    };

    // Hand unit u's slots back: issue the unit DEC_UNITS ahead into them and
    // load the page ids of the unit after that.
    auto release_unit = [&](int u, int st) {  // st = u % DEC_UNITS, also the slot group of u + DEC_UNITS
        __syncwarp();
        if (u + DEC_UNITS < n_units) {  // warp-uniform
            fence_proxy_async_smem();
            issue_unit(u + DEC_UNITS, st, pid_next);
            n_issued = u + DEC_UNITS + 1;
            const int j = UNIT_PAGES * (u + DEC_UNITS + 1) + lane;
            if (lane < UNIT_PAGES && j < my_count) pid_next = __ldg(bt + page_of(j));
        }
    };

    // Software pipeline over the warp's units: the QK of unit u + 1 does not
    // depend on the softmax or PV of unit u, and the two sit in one
    // straight-line block so their instruction streams interleave.
    // The slot group and mbarrier parity of unit u advance with u (no
    // division by the ring size in the loop).
    int u_fail = -1;  // the unit whose wait timed out
    float lg[UNIT_PAGES][NT][2], pm[NT];
    int st = 0;             // u % DEC_UNITS
    uint32_t parity = 0u;   // (u / DEC_UNITS) & 1
    if (n_units > 0) {
        if (wait_unit(0, 0u))
            qk_unit(0, lg, pm);
        else
            u_fail = 0;
    }
    int u = 0;
    for (; u + 1 < n_units && u_fail < 0; ++u) {
        const int st1 = st + 1 == DEC_UNITS ? 0 : st + 1;
        const uint32_t parity1 = st + 1 == DEC_UNITS ? parity ^ 1u : parity;
        float pr[UNIT_PAGES][NT][2];
        softmax_unit(lg, pm, pr);
        if (!wait_unit(st1, parity1)) {
            u_fail = u + 1;
            break;
        }
#pragma unroll
        for (int e = 0; e < UNIT_PAGES; ++e) pv_page(UNIT_PAGES * st + e, pr[e]);
        qk_unit(st1, lg, pm);  // lg, pm of unit u are spent (pr holds what PV needs)
        release_unit(u, st);
        st = st1;
        parity = parity1;
    }
    if (u_fail < 0 && n_units > 0) {
        float pr[UNIT_PAGES][NT][2];
        softmax_unit(lg, pm, pr);
#pragma unroll
        for (int e = 0; e < UNIT_PAGES; ++e) pv_page(UNIT_PAGES * st + e, pr[e]);
    }
    if (u_fail >= 0 && lane == 0) {
        // let copies still in flight land before the shared memory is reused
        for (int v = u_fail; v < n_issued; ++v)
            (void)mbar_wait_bounded(&sm.bar[warp][v % DEC_UNITS], (v / DEC_UNITS) & 1, 1000000LL);
    }

    // the next kernel in the stream may be scheduled once every CTA is here
    griddep_launch_dependents();

    // ---------------- warp partial -> shared memory
    __syncthreads();  // all warps are done with the ring (o_part aliases it)
    {
        // min term of (group g, head 2t / 2t+1) lives in lane 4g + t
        float cm[NGROUP][2];
#pragma unroll
        for (int g = 0; g < NGROUP; ++g) {
            cm[g][0] = __shfl_sync(0xffffffffu, cmin[0], 4 * g + t);
            cm[g][1] = __shfl_sync(0xffffffffu, cmin[1], 4 * g + t);
        }
        if constexpr (NT == 1) {
            // columns 4..7 (lanes t = 2, 3) hold the low parts of heads 0..3
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[m][e] += __shfl_xor_sync(0xffffffffu, oacc[m][e], 2);
        }
        const bool writer = NT == 2 || t < 2;
#pragma unroll
        for (int g = 0; g < NGROUP; ++g)
#pragma unroll
            for (int hs = 0; hs < 2; ++hs) {
                const int m = 2 * g + hs;
                const int ch0 = 32 * g + 4 * r + 2 * hs;     // row r, k = 2hs
                const float f0 = ldexpf(1.f, 24 - 4 * hs);  // 2^24 / 4^(2hs)
                const float f1 = f0 * 0.25f;                     // row r + 8, k = 2hs + 1
                if (writer && 2 * t < G) {
                    sm.u.o_part[warp][2 * t][ch0] = fmaf(oacc[m][0], f0, cm[g][0]);
                    sm.u.o_part[warp][2 * t][ch0 + 1] = fmaf(oacc[m][2], f1, cm[g][0]);
                }
                if (writer && 2 * t + 1 < G) {
                    sm.u.o_part[warp][2 * t + 1][ch0] = fmaf(oacc[m][1], f0, cm[g][1]);
                    sm.u.o_part[warp][2 * t + 1][ch0 + 1] = fmaf(oacc[m][3], f1, cm[g][1]);
                }
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float l = lsum[nt];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int hq = 4 * nt + t;
            if (r == 0 && hq < G) {
                sm.ms.m_part[warp][hq] = mrun[nt];
                sm.ms.l_part[warp][hq] = l;
            }
        }
    }
    __syncthreads();

    finish_decode<NW, MAXG>(sm.ms, sm.u.o_part, G, H_q, H_kv, B, b, h, split, S, ws, Rv + (size_t)h * D * D, out);
}

}  // namespace kvq

using namespace kvq;

// The dynamic shared memory opt-in is a per-device attribute of the kernel:
// set it on the first call on each device only.
static kvq_status set_smem_once(const void* fn, int bytes, int which) {
    static std::mutex mu;
    static bool done[64][4] = {};
    int dev = 0;
    kvq_status st = kvq_check_cuda(cudaGetDevice(&dev), "kvq_decode_attn_int2: cudaGetDevice");
    if (st != KVQ_OK) return st;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev][which]) return KVQ_OK;
    st = kvq_check_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                        "kvq_decode_attn_int2 smem attribute");
    if (st == KVQ_OK && dev >= 0 && dev < 64) done[dev][which] = true;
    return st;
}

extern "C" int kvq_decode_auto_splits(int B, int H_q, int H_kv, int max_pages_per_seq) {
    if (B <= 0 || H_kv <= 0 || H_q < H_kv || max_pages_per_seq <= 0) return 1;
    // at most one wave of CTAs, one per SM of the 152, over the (sequence,
    // KV head) pairs (a CTA past the wave would run alone in a second one);
    // at least 32 pages per split (the CTAs have 8-12 warps)
    const long units = (long)B * H_kv;
    long s = 152L / units;
    long max_s = (max_pages_per_seq + 31) / 32;
    if (max_s > MAX_SPLITS) max_s = MAX_SPLITS;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    return (int)s;
}

extern "C" size_t kvq_decode_workspace_bytes(int B, int H_q, int H_kv, int max_pages_per_seq, int num_splits) {
    if (B <= 0 || H_q <= 0 || H_kv <= 0) return 0;
    int S = num_splits;
    if (S <= 0) {  // room for the automatic choice of every decode entry point
        S = kvq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq) + 1;  // + 1: a BF16 window split
        const int Sb = bgtq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
        if (Sb > S) S = Sb;
    }
    return WS_HEADER + tickets_bytes(B, H_kv) + (size_t)B * H_q * S * PART_STRIDE * sizeof(float);
}

// Validation and launch shared by the two INT2 decode entry points; `win_k`
// null means no BF16 window.
static kvq_status decode_int2_launch(const char* fn, const void* q, int B, int H_q, int H_kv, int d,
                                     const void* cache, int64_t num_pages, const int32_t* block_table,
                                     int max_pages_per_seq, const int32_t* context_lens, const float* R_k,
                                     const float* R_v, const float* mu_k, const void* win_k, const void* win_v,
                                     const int32_t* win_lens, int win_max, float scale, float* out, void* workspace,
                                     size_t workspace_bytes, int num_splits, void* stream) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: d=%d (only 128)", fn, d);
    if (B <= 0 || H_kv <= 0 || H_q <= 0 || H_q % H_kv || max_pages_per_seq <= 0 || num_pages <= 0 ||
        num_splits < 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: B=%d H_q=%d H_kv=%d max_pages=%d num_pages=%lld splits=%d",
                             fn, B, H_q, H_kv, max_pages_per_seq, (long long)num_pages, num_splits);
    const int G = H_q / H_kv;
    if (G > 8) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: GQA group %d > 8", fn, G);
    if (B > 65535 || H_kv > 65535) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: B or H_kv above 65535", fn);
    if (!q || !cache || !block_table || !context_lens || !R_k || !R_v || !out || !workspace)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (reinterpret_cast<uintptr_t>(cache) % 16 || reinterpret_cast<uintptr_t>(workspace) % 16 ||
        reinterpret_cast<uintptr_t>(R_v) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: cache, R_v and workspace need 16-byte alignment", fn);
    if (win_k) {
        if (win_max <= 0 || !win_v || !win_lens || !mu_k)
            return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: window needs win_max > 0, win_v, win_lens and mu_k", fn);
        if (reinterpret_cast<uintptr_t>(win_k) % 16 || reinterpret_cast<uintptr_t>(win_v) % 16)
            return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: win_k and win_v need 16-byte alignment", fn);
    }
    int S_pages = num_splits > 0 ? num_splits : kvq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
    // the automatic choice fills one wave; with a window, its split takes
    // one of those CTAs (a 153rd CTA would run alone in a second wave)
    if (num_splits == 0 && win_k && S_pages > 1 && (long)(S_pages + 1) * B * H_kv > 152L) S_pages -= 1;
    const int S = S_pages + (win_k ? 1 : 0);
    if (S > MAX_SPLITS)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: %d splits above %d", fn, S, MAX_SPLITS);
    const size_t need = kvq_decode_workspace_bytes(B, H_q, H_kv, max_pages_per_seq, S);
    if (workspace_bytes < need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
    const float scale_log2 = scale * 1.4426950408889634f;
    constexpr int NW1 = DecWarps<1>::NW, NW2 = DecWarps<2>::NW;
    const size_t smem = G <= 4 ? sizeof(DecodeSmem<NW1, 4>) : sizeof(DecodeSmem<NW2, 8>);
    dim3 grid(S, H_kv, B);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto* kern = G <= 4 ? (win_k ? decode_int2_kernel<1, true> : decode_int2_kernel<1, false>)
                        : (win_k ? decode_int2_kernel<2, true> : decode_int2_kernel<2, false>);
    kvq_status sa = set_smem_once((const void*)kern, (int)smem, (G <= 4 ? 0 : 2) + (win_k ? 1 : 0));
    if (sa != KVQ_OK) return sa;
    const cudaError_t e =
        launch_pdl(kern, grid, dim3((G <= 4 ? NW1 : NW2) * 32), smem, st, static_cast<const __nv_bfloat16*>(q), H_q,
                   H_kv, G, static_cast<const uint8_t*>(cache), num_pages, block_table, max_pages_per_seq,
                   context_lens, R_k, R_v, mu_k, static_cast<const __nv_bfloat16*>(win_k),
                   static_cast<const __nv_bfloat16*>(win_v), win_lens, win_max, scale_log2, out,
                   static_cast<uint8_t*>(workspace));
    return kvq_check_cuda(e, "decode launch");
}

extern "C" kvq_status kvq_decode_attn_int2(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                           int64_t num_pages, const int32_t* block_table, int max_pages_per_seq,
                                           const int32_t* context_lens, const float* R_k, const float* R_v,
                                           float scale, float* out, void* workspace, size_t workspace_bytes,
                                           int num_splits, void* stream) {
    return decode_int2_launch("kvq_decode_attn_int2", q, B, H_q, H_kv, d, cache, num_pages, block_table,
                              max_pages_per_seq, context_lens, R_k, R_v, nullptr, nullptr, nullptr, nullptr, 0, scale,
                              out, workspace, workspace_bytes, num_splits, stream);
}

extern "C" kvq_status kvq_decode_attn_int2_window(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                                  int64_t num_pages, const int32_t* block_table,
                                                  int max_pages_per_seq, const int32_t* context_lens,
                                                  const float* R_k, const float* R_v, const float* mu_k,
                                                  const void* win_k, const void* win_v, const int32_t* win_lens,
                                                  int win_max, float scale, float* out, void* workspace,
                                                  size_t workspace_bytes, int num_splits, void* stream) {
    if (!win_k) return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_decode_attn_int2_window: null win_k");
    return decode_int2_launch("kvq_decode_attn_int2_window", q, B, H_q, H_kv, d, cache, num_pages, block_table,
                              max_pages_per_seq, context_lens, R_k, R_v, mu_k, win_k, win_v, win_lens, win_max, scale,
                              out, workspace, workspace_bytes, num_splits, stream);
}

extern "C" kvq_status kvq_workspace_status(void* workspace, void* stream) {
    if (!workspace) return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_workspace_status: null workspace");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    kvq_status s = kvq_check_cuda(cudaMemcpyAsync(&word, workspace, 4, cudaMemcpyDeviceToHost, st), "status read");
    if (s != KVQ_OK) return s;
    s = kvq_check_cuda(cudaStreamSynchronize(st), "status sync");
    if (s != KVQ_OK) return s;
    if (word) {
        s = kvq_check_cuda(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
        if (s != KVQ_OK) return s;
        s = kvq_check_cuda(cudaStreamSynchronize(st), "status clear sync");
        if (s != KVQ_OK) return s;
    }
    if (word & ERR_TIMEOUT) return kvq_set_error(KVQ_ERR_CUDA, "decode: an in-kernel wait timed out");
    if (word & ERR_BAD_WIDTHS) return kvq_set_error(KVQ_ERR_INVALID_ARG, "decode: widths outside 1..8 or over budget");
    if (word & ERR_BAD_PAGE) return kvq_set_error(KVQ_ERR_BAD_BLOCK_TABLE, "decode: block table entry out of range");
    return KVQ_OK;
}
