// Fused packed-cache decode attention over the rotated INT2 cache.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization" §3 Eqs. (1)-(2)
// with Eq. (4) folded in: <q, Q2(zR)R^T> = <qR, Q2(zR)>, so the query is
// rotated once (q' = q R_k), the cache is consumed in the rotated basis and
// the output is rotated back once (o = o' R_v^T).  The kernel reads only the
// packed codes and fp16 (scale, min) pairs.
//
// One large CTA per SM of 12 warps.  The batch's (sequence, KV head) units are laid end to end as virtual
// pages and every CTA takes an equal contiguous share (at most two units),
// so all SMs stream whatever B * H_kv is; within a share the pages are dealt
// round-robin over the CTA's warps.  Each warp streams pages through its own
// ring of 1536-byte tiles (9 slots for head groups up to 4, 6 for groups of
// 8) filled by bulk async copies (cp.async.bulk + mbarrier).  Per page (16
// tokens):
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
// Each CTA merges its warps, rotates the merged partial by R_v^T (linear,
// so this equals one rotation of the final output) and publishes it per
// unit; the last CTA of a (sequence, KV head) to finish (atomic ticket, no
// waiting) merges the unit's partials and writes the output.  In the decode
// step the CTA holding a sequence's new token also quantises and writes it,
// and attends it from registers.
#include <atomic>
#include <mutex>

#include "int2_quant.cuh"
#include "merge.cuh"

namespace kvq {

constexpr int UNIT_PAGES = 3;  // pages per mbarrier phase (one wait, one release)

// Page slots per warp: 9 (three units in flight) for head groups up to 4;
// 6 for groups of 8, whose twelve warps would not fit 227 KB with nine.
template <int MAXG>
struct DecRing {
    static constexpr int STAGES = MAXG <= 4 ? 9 : 6;
    static constexpr int UNITS = STAGES / UNIT_PAGES;
    static_assert(STAGES % UNIT_PAGES == 0, "a unit is a whole number of page slots");
};

// Warps per CTA: twelve, three per scheduler at 168 registers (a quarter of
// the SM's 64K registers each).  Groups of 8 keep their QK B fragments in
// shared memory (for 4 heads they stay in registers) to fit that budget.
template <int NT>
struct DecWarps {
    static constexpr int NW = 12;
};

template <int NW, int MAXG>
struct __align__(16) DecodeSmem {
    struct {
        uint8_t ring[NW][DecRing<MAXG>::STAGES][INT2_TILE];  // page tiles in flight
    } u;
    float o_part[NW + 1][MAXG][D];  // per-warp o' after the loop (its own space: a warp writes it as soon as
                                    // it is done), and the decode step's new token
    uint64_t bar[NW][DecRing<MAXG>::UNITS];
    int ntok[NW][DecRing<MAXG>::STAGES];  // valid tokens of the page in each stage (0: skipped page)
    float q[MAXG][D];          // scaled rotated queries q~ = q R_k * scale * log2(e)
    float gsum[MAXG][NGROUP];
    float sigma[MAXG];         // power-of-two pre-scale per head
    int64_t share[2];          // this CTA's virtual pages [share[0], share[1])
    int dead;                  // a wait of this CTA ran out: no further copies
    uint2 bq[MAXG == 8 ? 2 : 1][8][32];  // groups of 8: QK B fragments (n-tile, k-slice, lane)
    MergeSmem<NW, MAXG> ms;
};

static_assert(sizeof(DecodeSmem<12, 4>) <= 227 * 1024 && sizeof(DecodeSmem<12, 8>) <= 227 * 1024,
              "decode shared memory above 227 KB");

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
    // The warp's tokens t = warp, warp + NW, ... in chunks of WC: a chunk's
    // WC x MAXG dot products are independent, so their shuffle reductions
    // overlap (every head is computed; heads past G have q = 0), and the
    // chunk joins the running softmax with one maximum update.  The next
    // chunk's rows are requested before this one is computed.  Rows past
    // the window are clamped to its last row (a valid address) and masked.
    constexpr int WC = MAXG == 8 ? 2 : 4;  // (registers: groups of 8 hold twice the heads)
    auto load_chunk = [&](int t0, uint2 (&kr)[WC], uint2 (&vr)[WC]) {
#pragma unroll
        for (int i = 0; i < WC; ++i) {
            const size_t row = (((size_t)b * win_max + min(t0 + i * NW, wl - 1)) * H_kv + h) * D + 4 * lane;
            kr[i] = __ldg(reinterpret_cast<const uint2*>(win_k + row));
            vr[i] = __ldg(reinterpret_cast<const uint2*>(win_v + row));
        }
    };
    uint2 kn[WC], vn[WC];
    if (warp < wl) load_chunk(warp, kn, vn);
#pragma unroll 1
    for (int t0 = warp; t0 < wl; t0 += WC * NW) {
        uint2 kr[WC], vr[WC];
#pragma unroll
        for (int i = 0; i < WC; ++i) {
            kr[i] = kn[i];
            vr[i] = vn[i];
        }
        if (t0 + WC * NW < wl) load_chunk(t0 + WC * NW, kn, vn);
        float lg[WC][MAXG];
#pragma unroll
        for (int i = 0; i < WC; ++i) {
            const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kr[i].x));
            const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kr[i].y));
            const float kc[4] = {__fsub_rn(k01.x, mc[0]), __fsub_rn(k01.y, mc[1]), __fsub_rn(k23.x, mc[2]),
                                 __fsub_rn(k23.y, mc[3])};
#pragma unroll
            for (int jj = 0; jj < MAXG; ++jj) {
                float dot = qv[jj][0] * kc[0];
#pragma unroll
                for (int e = 1; e < 4; ++e) dot = fmaf(qv[jj][e], kc[e], dot);
                lg[i][jj] = dot;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int i = 0; i < WC; ++i)
#pragma unroll
                for (int jj = 0; jj < MAXG; ++jj) lg[i][jj] += __shfl_xor_sync(0xffffffffu, lg[i][jj], o);
#pragma unroll
        for (int jj = 0; jj < MAXG; ++jj) {
            // token t0 is in the window, so the chunk's maximum is finite
            float mn = m_w[jj];
#pragma unroll
            for (int i = 0; i < WC; ++i) {
                lg[i][jj] = t0 + i * NW < wl ? lg[i][jj] * scale_log2 : -CUDART_INF_F;
                mn = fmaxf(mn, lg[i][jj]);
            }
            const float corr = ex2(m_w[jj] - mn);  // 0 while nothing was seen
            float ps = 0.f, ov[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < WC; ++i) {
                const float p = ex2(lg[i][jj] - mn);  // 0 for a masked row
                const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr[i].x));
                const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr[i].y));
                ps += p;
                ov[0] = fmaf(p, v01.x, ov[0]);
                ov[1] = fmaf(p, v01.y, ov[1]);
                ov[2] = fmaf(p, v23.x, ov[2]);
                ov[3] = fmaf(p, v23.y, ov[3]);
            }
            l_w[jj] = fmaf(l_w[jj], corr, ps);
#pragma unroll
            for (int e = 0; e < 4; ++e) o_w[jj][e] = fmaf(o_w[jj][e], corr, ov[e]);
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

// Work split.  The B * H_kv (sequence, KV head) units are laid end to end
// as V = units * vmp "virtual" pages (vmp = max_pages, plus in a decode step
// or a window decode a few pages without work after the real ones, which
// lighten the share holding the new token or attending the window):
// unit u = b * H_kv + h owns
// [u * MP, (u + 1) * MP), of which the first ceil(ctx_b / 16) are real.
// Page CTA c of C takes the virtual pages [c V / C, (c + 1) V / C), so every
// CTA gets the same share (within one page) whatever B * H_kv is, and a CTA
// whose share crosses a unit boundary works on each unit in turn (a
// segment).  The CTAs that touch unit u are cta_of(u MP) .. cta_of(u MP +
// MP - 1); each publishes one partial in slot u + c (unique: the shares are
// ordered), and the one that arrives last merges them.  Needs 1 <= C <= V.
struct PageSplit {
    int64_t V;
    int C, MP;
    __device__ __forceinline__ int64_t start(int c) const { return (int64_t)c * V / C; }
    __device__ __forceinline__ int cta_of(int64_t g) const { return (int)(((g + 1) * C - 1) / V); }
};

// What a decode attends besides the cached pages of a (sequence, KV head) unit.
enum DecodeMode : int {
    MODE_CACHE = 0,   // nothing: the cache alone
    MODE_WINDOW = 1,  // the unit's BF16 window
    MODE_STEP = 2,    // append the decode token to the cache and attend it
};

// The new token of a decode step (MODE_STEP), KV head h of sequence b, at
// position ctx - 1: quantised exactly as the append kernels do it (the same
// fp32 chains z = (k - mu) R_k, w = v R_v in ascending input order, the same
// group parameters and codes) and written to its cache slot.  The CTA whose
// page share holds that position does it, between issuing its first copies
// and rotating the query; its first 256 threads work (thread j < 128 owns
// rotated key channel j, thread 128 + j value channel j) on inputs staged in
// xs[0] (centred key) and xs[1] (value).  Returns the level the cache now
// holds for the thread's channel (0 for other threads), so the token can be
// attended from registers.
__device__ __forceinline__ float new_token_codes(const float (*xs)[D], const float (&rcol)[D], uint8_t* __restrict__ cache,
                                                 int H_kv, int h, int pid, int slot, bool write) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int side = tid >> 7;
    if (tid >= 2 * D) return 0.f;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) acc = __fmaf_rn(xs[side][i], rcol[i], acc);
    // group parameters (exact min / max over the 32 lanes of the group)
    float mn = acc, mx = acc;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    __half sh, mh;
    int2_params(mn, mx, 1.f, sh, mh);
    const float scf = __half2float(sh), mnf = __half2float(mh);
    const int code = int2_code(acc, mnf, scf);
    const uint32_t byte = int2_gather_byte(code, lane);
    const int grp = warp & 3;
    if (write) {
        uint8_t* tile = cache + ((size_t)pid * H_kv + h) * INT2_TILE;
        if ((lane & 3) == 0) tile[(side ? OFF_VC : OFF_KC) + 32 * slot + 4 * (lane >> 2) + grp] = (uint8_t)byte;
        if (lane == 0) int2_store_meta(tile, side, slot, grp, sh, mh);
    }
    return fmaf((float)code, scf, mnf);
}

// The new token as one more row of this CTA's warp partials: logit
// q~ . k^ per head (q~ the rotated, scaled query in qt, k^ held by threads
// j < 128), l = 1, o' = v^ (threads 128 + j, rotated basis); an empty row when
// the token was not written.  fac is scratch [MAXG][>= 4].  All threads call
// it; it ends with a barrier.
template <int NW, int MAXG>
__device__ __forceinline__ void new_token_row(MergeSmem<NW, MAXG>& ms, float (*o_row)[D], const float (*qt)[D],
                                              float xhat, bool ok, int G) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int jj = 0; jj < MAXG; ++jj) {
        float v = (tid < D && jj < G) ? qt[jj][tid] * xhat : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && warp < 4) ms.fac[jj][warp] = v;
    }
    if (tid >= D && tid < 2 * D) {
        for (int jj = 0; jj < G; ++jj) o_row[jj][tid - D] = ok ? xhat : 0.f;
    }
    __syncthreads();
    if (tid < G) {
        ms.m_part[NW][tid] = ok ? ms.fac[tid][0] + ms.fac[tid][1] + ms.fac[tid][2] + ms.fac[tid][3] : -CUDART_INF_F;
        ms.l_part[NW][tid] = ok ? 1.f : 0.f;
    }
    __syncthreads();
}

// Test hook: CTA 0 leaves the bulk copy of its first page unissued (the unit
// is still armed with its bytes), so that wait runs out after a short limit.
constexpr int DBG_DROP_FIRST_COPY = 1;
// The caller declares that the rotations, key centre, block table, context
// lengths and cache are not written by the kernel just before: the first
// segment's page ids, first copies and rows of R_k then go out before the
// dependency wait (the query, the new token and the workspace are only read
// or written after it).
constexpr int FLAG_EARLY_INPUTS = 2;
constexpr long long DBG_WAIT_LIMIT_CYCLES = 2000000LL;

// Grid: n_cta page CTAs.  In MODE_WINDOW the CTA whose share holds a unit's
// last virtual page also attends that unit's BF16 window, after its pages,
// and publishes it as one more partial of the unit.  In MODE_STEP, k_new / v_new are the decode token's [B][H_kv][d] key
// and value (win_k and win_v carry them), appended at position ctx - 1 by the
// page CTA whose share holds that position.
template <int NT, int MODE>
__global__ void __launch_bounds__(DecWarps<NT>::NW * 32, 1)
decode_int2_kernel(const __nv_bfloat16* __restrict__ q, int B, int H_q, int H_kv, int G,
                   uint8_t* __restrict__ cache, int64_t num_pages, const int32_t* __restrict__ block_table,
                   int max_pages, const int32_t* __restrict__ context_lens, const float* __restrict__ Rk,
                   const float* __restrict__ Rv, const float* __restrict__ mu,
                   const __nv_bfloat16* __restrict__ win_k, const __nv_bfloat16* __restrict__ win_v,
                   const int32_t* __restrict__ win_lens, int win_max, float scale_log2, float* __restrict__ out,
                   uint8_t* __restrict__ ws, int n_cta, int vmp, int flags) {
    constexpr int DEC_STAGES = DecRing<4 * NT>::STAGES;  // page slots per warp
    constexpr int DEC_UNITS = DecRing<4 * NT>::UNITS;    // units in flight per warp
    constexpr bool WIN = MODE == MODE_WINDOW;  // each unit has a window partial besides the page CTAs' ones
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int MAXG = 4 * NT;
    constexpr int NW = DecWarps<NT>::NW;
    DecodeSmem<NW, MAXG>& sm = *reinterpret_cast<DecodeSmem<NW, MAXG>*>(smem_raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane >> 2, t = lane & 3;
    // The workspace pointers and the split are formed where they are used
    // (from the kernel parameters), so the page loop holds no registers for
    // them.
    auto slot_ptr = [&](int64_t slot) {
        float* partials = reinterpret_cast<float*>(ws + WS_HEADER + tickets_bytes(B, H_kv));
        return partials + (size_t)slot * G * PART_STRIDE;
    };
    // Each unit's partials are one CTA's alone (one page CTA per unit, no
    // window): then no slot, ticket or merge is needed.  The shares are
    // equal, so a unit has a single CTA exactly when there are as many CTAs
    // as units (with more CTAs every share is shorter than a unit).  Groups
    // of 8 keep the merge path: with the direct one compiled in, their
    // batch-32 128K decode ran 4.7 % slower (register allocation).
    const bool sole = NT == 1 && !WIN && n_cta == B * H_kv;
    auto finish_unit = [&](int u) {
        // publish this CTA's slot (already written), then the last CTA merges;
        // the partials of unit u are the page CTAs' slots u + c, then (with a
        // window) the window's slot units + n_cta + u
        const PageSplit sp{(int64_t)B * H_kv * vmp, n_cta, vmp};
        const int units = B * H_kv;
        const int c0 = sp.cta_of((int64_t)u * vmp);
        const int n = sp.cta_of((int64_t)u * vmp + vmp - 1) - c0 + 1;
        const int expected = n + (WIN ? 1 : 0);
        int32_t* tickets = reinterpret_cast<int32_t*>(ws + WS_HEADER);
        if (!arrive_last(sm.ms, tickets + u, expected)) return;
        const int b = u / H_kv, h = u % H_kv;
        auto slot_of = [&](int s) -> const float* {
            return s < n ? slot_ptr((int64_t)u + c0 + s) : slot_ptr((int64_t)units + n_cta + u);
        };
        merge_out<NW, MAXG>(sm.ms, slot_of, expected, G, out + ((size_t)b * H_q + (size_t)h * G) * D);
        if (tid == 0) tickets[u] = 0;
    };

    const int cta = blockIdx.x;
    int u_first;
    {
        const PageSplit sp{(int64_t)B * H_kv * vmp, n_cta, vmp};
        const int64_t g0 = sp.start(cta);
        u_first = (int)(g0 / vmp);
        if (tid == 0) {
            // the share bounds live in shared memory, so the page loop below
            // holds no registers for them
            sm.share[0] = g0;
            sm.share[1] = sp.start(cta + 1);
            sm.dead = 0;
        }
        // the ring's mbarriers are set up once: a warp's units keep one
        // numbering across the segments (slot group k % 3, parity (k / 3) & 1)
        if (lane == 0) {
            for (int s2 = 0; s2 < DEC_UNITS; ++s2) mbar_init(&sm.bar[warp][s2], 1);
            fence_mbar_init();
        }
        // Prefetches into L2 only (a prefetch returns no data, and L2 is the
        // point of coherence, so a write the previous kernel makes later
        // still wins): the first unit's rotations, context length and query
        // rows, and this warp's first block-table entries.
        const int b = u_first / H_kv, h = u_first % H_kv;
        const char* rk = reinterpret_cast<const char*>(Rk + (size_t)h * D * D);
        const char* rv = reinterpret_cast<const char*>(Rv + (size_t)h * D * D);
        for (int l = tid; l < D * D * 4 / 128; l += NW * 32) {
            prefetch_l2(rk + 128 * l);
            prefetch_l2_keep(rv + 128 * l);
        }
        const int pa = (int)(g0 - (int64_t)u_first * vmp);
        const int j = pa + warp + NW * lane;
        if (lane < DEC_STAGES + UNIT_PAGES && j < max_pages) prefetch_l2(block_table + (size_t)b * max_pages + j);
        if (tid == 0) prefetch_l2(context_lens + b);
        const char* qc = reinterpret_cast<const char*>(q + ((size_t)b * H_q + (size_t)h * G) * D);
        if (tid < (G * D * 2 + 127) / 128) prefetch_l2(qc + 128 * tid);
    }
    const bool early = flags & FLAG_EARLY_INPUTS;
    if (!early) griddep_wait();  // every input may come from the previous kernel in the stream
    __syncthreads();             // the share bounds are in shared memory

    constexpr int QPT = (MAXG * D + NW * 32 - 1) / (NW * 32);  // query values per thread
    int kbase = 0;  // units this warp consumed in earlier segments

    // One segment: the part of this CTA's share that lies in unit u.  A share
    // spans at most two units (the host keeps C >= B * H_kv), so the body is
    // expanded twice instead of looped: no loop-carried state competes with
    // the page loop for registers.
    auto segment = [&](int u, bool second) {
        const int b = u / H_kv, h = u % H_kv;
        const int64_t ubase = (int64_t)u * vmp;
        const int64_t g0 = sm.share[0], g1 = sm.share[1];
        const bool last_seg = g1 <= ubase + vmp;  // this CTA's share ends in unit u
        // the share's pages of unit u: [pa, pb) of its vmp virtual pages (the
        // pages past max_pages, a decode step's balance, carry no work)
        const int pa = (int)(max(g0, ubase) - ubase), pb = (int)(min(g1, ubase + vmp) - ubase);
        const int32_t* bt = block_table + (size_t)b * max_pages;
        // pages pa .. pe - 1 of the unit (pe: the share's end or the context's),
        // dealt round-robin over the warps
        auto page_of = [&](int j) { return pa + warp + NW * j; };
        // The loads the prologue needs all go out together: the context length,
        // (lanes 0..2) the page ids of the warp's first units -- bounded by the
        // share, not the context, so they need not wait for its length -- this
        // warp's rows of R_k and the query values.
        int ctx = __ldg(context_lens + b);
        int pid_first[DEC_UNITS];
        int pid_next = 0;
        {
            const int cs = min(pb, max_pages) - pa, my_share = cs > warp ? (cs - warp + NW - 1) / NW : 0;
#pragma unroll
            for (int k = 0; k < DEC_UNITS; ++k) pid_first[k] = 0;
            if (lane < UNIT_PAGES) {
#pragma unroll
                for (int k = 0; k <= DEC_UNITS; ++k) {
                    const int j = UNIT_PAGES * k + lane;
                    const int pid = j < my_share ? __ldg(bt + page_of(j)) : 0;
                    if (k < DEC_UNITS)
                        pid_first[k] = pid;
                    else
                        pid_next = pid;
                }
            }
        }
        ctx = max(0, min(ctx, max_pages * PAGE));
        // the decode step's new token sits at position ctx - 1: the pages hold
        // the ctx - 1 tokens before it, and the CTA whose share holds its page
        // quantises, writes and attends it
        const int ctx_all = ctx;
        if (MODE == MODE_STEP) ctx = max(ctx - 1, 0);
        const int p_new = (ctx_all - 1) / PAGE;
        const bool has_new = MODE == MODE_STEP && ctx_all > 0 && p_new >= pa && p_new < pb;
        const int n_pages = (ctx + PAGE - 1) / PAGE;
        const int pe = min(pb, n_pages);
        // no cached page of this unit in this CTA's share (or a wait ran out
        // earlier): nothing to stream
        const bool empty = pe <= pa || sm.dead;
        if (!empty || has_new) {
        const int count = empty ? 0 : pe - pa;
        const int my_count = count > warp ? (count - warp + NW - 1) / NW : 0;

        float4 rr[RowPrefetch<NW, MAXG>::N];
        if constexpr (MODE != MODE_STEP) load_rows<NW>(Rk + (size_t)h * D * D, rr);
        float qv[QPT];
        auto load_q = [&]() {
            const __nv_bfloat16* qb = q + ((size_t)b * H_q + (size_t)h * G) * D;
#pragma unroll
            for (int k = 0; k < QPT; ++k) {
                const int idx = tid + k * NW * 32;
                qv[k] = idx < G * D ? __bfloat162float(qb[idx]) : 0.f;
            }
        };
        if (!early) load_q();
        const int n_units = (my_count + UNIT_PAGES - 1) / UNIT_PAGES;
        __syncwarp();
        // in a second segment the ring was last read through the generic
        // proxy: order that before the bulk copies any lane issues
        if (second) fence_proxy_async_smem();
        // slot group and parity of this segment's first unit
        const int st0 = kbase % DEC_UNITS;
        const uint32_t par0 = (kbase / DEC_UNITS) & 1;

        // Lanes e < UNIT_PAGES issue page e of unit k (id pid) into slot group
        // st and record how many tokens of it are valid (0 for a slot past the
        // warp's pages or with a bad page id); the mbarrier publishes the
        // counts with the data.
        auto issue_unit = [&](int k, int st, int pid) {
            uint64_t* bar = &sm.bar[warp][st];
            const int j = UNIT_PAGES * k + lane;
            bool ok = false;
            if (lane < UNIT_PAGES) {
                int n = 0;
                if (j < my_count) {
                    if (pid < 0 || (int64_t)pid >= num_pages) {
                        atomicOr(reinterpret_cast<uint32_t*>(ws), ERR_BAD_PAGE);
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
            // (test hook: CTA 0 leaves its first copy unissued)
            if (ok && !((flags & DBG_DROP_FIRST_COPY) && cta == 0 && warp == 0 && u == 0 && k == 0 && lane == 0))
                bulk_g2s_hint(sm.u.ring[warp][UNIT_PAGES * st + lane], cache + ((size_t)pid * H_kv + h) * INT2_TILE,
                              INT2_TILE, bar, l2_policy_evict_first());
        };
        // the first units go out as soon as their page ids are here: the copies
        // fly while the query is rotated
        int n_issued = 0;
#pragma unroll
        for (int k = 0; k < DEC_UNITS; ++k)
            if (k < n_units) {  // warp-uniform
                issue_unit(k, st0 + k < DEC_UNITS ? st0 + k : st0 + k - DEC_UNITS, pid_first[k]);
                n_issued = k + 1;
            }
        // the rest of this share of the block table is read one entry at a
        // time during the loop: have L2 fetch it now (every address is an
        // entry of the share, so no line past the table is touched)
        for (int i = pa + 32 * tid; i < pa + count + 31; i += 32 * NW * 32) prefetch_l2_keep(bt + min(i, pe - 1));
        float xhat = 0.f;  // (decode step) the new token's level in this thread's channel
        bool new_ok = false;
        if constexpr (MODE == MODE_STEP) {
            if (has_new) {  // CTA-uniform
                const int tsl = (ctx_all - 1) % PAGE;
                float rcol[D];
                if (tid < 2 * D) {
                    const float* R = (tid < D ? Rk : Rv) + (size_t)h * D * D + (tid & (D - 1));
#pragma unroll
                    for (int i = 0; i < D; ++i) rcol[i] = __ldg(R + (size_t)i * D);
                }
                const int pid_new = __ldg(bt + p_new);
                new_ok = pid_new >= 0 && (int64_t)pid_new < num_pages;
                if (early) griddep_wait();  // the new token comes from the previous kernel
                if (tid < D) {
                    const size_t row = ((size_t)b * H_kv + h) * D + tid;
                    sm.q[0][tid] = __fsub_rn(__bfloat162float(win_k[row]), __ldg(mu + (size_t)h * D + tid));
                    sm.q[1][tid] = __bfloat162float(win_v[row]);
                }
                __syncthreads();
                xhat = new_token_codes(sm.q, rcol, cache, H_kv, h, pid_new, tsl, new_ok);
                if (!new_ok && tid == 0) atomicOr(reinterpret_cast<uint32_t*>(ws), ERR_BAD_PAGE);
            }
            // the rows of R_k for the query rotation (after the new token's
            // columns, so the two never hold registers at once)
            load_rows<NW>(Rk + (size_t)h * D * D, rr);
        }
        if (early) {
            // the early inputs are out; the query may come from the previous kernel
            griddep_wait();
            load_q();
        }

        // ---- q~ = (q R_k) * scale * log2(e) for the G heads of this KV head
#pragma unroll
        for (int k = 0; k < QPT; ++k) {
            const int idx = tid + k * NW * 32;
            if (idx < G * D) sm.ms.o_final[idx / D][idx % D] = qv[k];
        }
        __syncthreads();
        rotate_rows<NW, MAXG>(sm.ms.o_final, Rk + (size_t)h * D * D, rr, G, scale_log2, sm.q, sm.ms);
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

        // ---- QK B fragments: column n = r -> head 4*nt + (r >> 1), part r & 1 (hi / lo)
        uint32_t bq[8][2];  // NT == 1: the fragments in registers (NT == 2: sm.bq)
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
                    const uint32_t w = pack_half2(lo_part ? v0 - h0 : h0, lo_part ? v1 - h1 : h1);
                    if constexpr (NT == 1) {
                        bq[s][e] = w;
                    } else if (warp == 0) {  // the same for every warp: one writes them
                        if (e == 0)
                            sm.bq[nt][s][lane].x = w;
                        else
                            sm.bq[nt][s][lane].y = w;
                    }
                }
            }
        }
        if constexpr (NT == 2) __syncthreads();  // the shared B fragments are complete
        float inv_sig[NT], gsum[NT][NGROUP];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hq = 4 * nt + t;
            inv_sig[nt] = hq < G ? 16777216.f / sm.sigma[hq] : 0.f;
#pragma unroll
            for (int g = 0; g < NGROUP; ++g) gsum[nt][g] = hq < G ? sm.gsum[hq][g] : 0.f;
        }

        if constexpr (MODE == MODE_STEP) {
            if (has_new) new_token_row<NW, MAXG>(sm.ms, sm.o_part[NW], sm.q, xhat, new_ok, G);
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

        // Wait for the unit in slot group st; false on a timeout.  On a
        // sequence's last page the slots past the context may hold stale bytes
        // (even NaN scales), and so does a slot with no page: their value
        // scale/min words are zeroed here, so p = 0 always meets finite factors
        // and the PV step needs no per-slot masks (the QK step drops those
        // slots' logits by selection).
        auto wait_unit = [&](int st, uint32_t parity) -> bool {
            const bool ok = mbar_wait_bounded(&sm.bar[warp][st], parity,
                                              (flags & DBG_DROP_FIRST_COPY) ? DBG_WAIT_LIMIT_CYCLES : WAIT_LIMIT_CYCLES);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) atomicOr(reinterpret_cast<uint32_t*>(ws), ERR_TIMEOUT);
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
                        if constexpr (NT == 1) {
                            mma_f16_16816(c, a, bq[2 * g + hs][0], bq[2 * g + hs][1]);
                        } else {
                            const uint2 bb = sm.bq[nt][2 * g + hs][lane];
                            mma_f16_16816(c, a, bb.x, bb.y);
                        }
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

        // QK of a unit and each head's maximum over its pages
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
        auto softmax_unit = [&](const float (&lg)[UNIT_PAGES][NT][2], const float (&pm)[NT],
                                float (&pr)[UNIT_PAGES][NT][2]) {
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
                // p^ * scale as an fp16 pair: hi = rn(p^ s), lo = p^ s - hi (exact).
                // Groups of 4 carry lo in the spare columns 4..7 (no extra MMA);
                // groups of 8 fill all eight columns with heads and take hi
                // alone: one rounding of p^ s to fp16 (relative error at most
                // 2^-11 per term, independent in sign across tokens) instead
                // of a second MMA per step.
                const __half2 S01 = u32_as_h2(wA[g]), S89 = u32_as_h2(wB[g]);
                const __half2 H0 = __hmul2(P0, S01), H1 = __hmul2(P1, S89);
#pragma unroll
                for (int hs = 0; hs < 2; ++hs) {
                    const uint32_t k0 = 0x00030003u << (4 * hs), k1 = 0x00030003u << (4 * hs + 2);
                    const uint32_t a[4] = {xa & k0, xa & k1, xb & k0, xb & k1};
                    if constexpr (NT == 1) {
                        const __half2 L0 = __hfma2(P0, S01, __hneg2(H0)), L1 = __hfma2(P1, S89, __hneg2(H1));
                        const bool lo = r >= 4;
                        mma_f16_16816(oacc[2 * g + hs], a, h2_as_u32(lo ? L0 : H0), h2_as_u32(lo ? L1 : H1));
                    } else {
                        mma_f16_16816(oacc[2 * g + hs], a, h2_as_u32(H0), h2_as_u32(H1));
                    }
                }
            }
        };

        // Hand unit k's slots back: issue the unit DEC_UNITS ahead into them and
        // load the page ids of the unit after that.
        auto release_unit = [&](int k, int st) {  // st = k % DEC_UNITS, also the slot group of k + DEC_UNITS
            __syncwarp();
            if (k + DEC_UNITS < n_units) {  // warp-uniform
                fence_proxy_async_smem();
                issue_unit(k + DEC_UNITS, st, pid_next);
                n_issued = k + DEC_UNITS + 1;
                const int j = UNIT_PAGES * (k + DEC_UNITS + 1) + lane;
                if (lane < UNIT_PAGES && j < my_count) pid_next = __ldg(bt + page_of(j));
            }
        };

        // Software pipeline over the warp's units: the QK of unit k + 1 does not
        // depend on the softmax or PV of unit k, and the two sit in one
        // straight-line block so their instruction streams interleave.  The
        // slot group and mbarrier parity advance with k (no division by the
        // ring size in the loop).
        int k_fail = -1;  // the unit whose wait timed out
        float lg[UNIT_PAGES][NT][2], pm[NT];
        int st = st0;           // (kbase + k) % DEC_UNITS
        uint32_t parity = par0;  // ((kbase + k) / DEC_UNITS) & 1
        if (n_units > 0) {
            if (wait_unit(st, parity))
                qk_unit(st, lg, pm);
            else
                k_fail = 0;
        }
        int k = 0;
        for (; k + 1 < n_units && k_fail < 0; ++k) {
            const int st1 = st + 1 == DEC_UNITS ? 0 : st + 1;
            const uint32_t parity1 = st + 1 == DEC_UNITS ? parity ^ 1u : parity;
            float pr[UNIT_PAGES][NT][2];
            softmax_unit(lg, pm, pr);
            if (!wait_unit(st1, parity1)) {
                k_fail = k + 1;
                break;
            }
#pragma unroll
            for (int e = 0; e < UNIT_PAGES; ++e) pv_page(UNIT_PAGES * st + e, pr[e]);
            qk_unit(st1, lg, pm);  // lg, pm of unit k are spent (pr holds what PV needs)
            release_unit(k, st);
            st = st1;
            parity = parity1;
        }
        if (k_fail < 0 && n_units > 0) {
            float pr[UNIT_PAGES][NT][2];
            softmax_unit(lg, pm, pr);
#pragma unroll
            for (int e = 0; e < UNIT_PAGES; ++e) pv_page(UNIT_PAGES * st + e, pr[e]);
        }
        if (k_fail >= 0) {
            if (lane == 0) {
                sm.dead = 1;
                // let copies still in flight land before the shared memory is reused
                for (int v = k_fail; v < n_issued; ++v)
                    (void)mbar_wait_bounded(&sm.bar[warp][(kbase + v) % DEC_UNITS], ((kbase + v) / DEC_UNITS) & 1,
                                            1000000LL);
            }
        }


        // the rows of R_v this warp rotates the CTA's partial with: loaded now,
        // so their latency passes during the merge of the warps
        float4 rvr[RowPrefetch<NW, MAXG>::N];
        load_rows<NW>(Rv + (size_t)h * D * D, rvr);
        // ---------------- warp partial -> shared memory, as soon as this warp is done
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
                    const float f1 = f0 * 0.25f;                 // row r + 8, k = 2hs + 1
                    if (writer && 2 * t < G) {
                        sm.o_part[warp][2 * t][ch0] = fmaf(oacc[m][0], f0, cm[g][0]);
                        sm.o_part[warp][2 * t][ch0 + 1] = fmaf(oacc[m][2], f1, cm[g][0]);
                    }
                    if (writer && 2 * t + 1 < G) {
                        sm.o_part[warp][2 * t + 1][ch0] = fmaf(oacc[m][1], f0, cm[g][1]);
                        sm.o_part[warp][2 * t + 1][ch0 + 1] = fmaf(oacc[m][3], f1, cm[g][1]);
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
        if (MODE == MODE_STEP && has_new)
            merge_warps<NW, MAXG, NW + 1>(sm.ms, sm.o_part, G);
        else
            merge_warps<NW, MAXG>(sm.ms, sm.o_part, G);
        kbase += n_units;
        // the next kernel in the stream may be scheduled once every CTA is here
        if (last_seg) griddep_launch_dependents();
        // this CTA's partial, carried to the output basis (O = o' R_v^T); a
        // unit whose only partial this is gets its output written directly
        rotate_publish<NW, MAXG>(sm.ms, rvr, G, Rv + (size_t)h * D * D,
                                 sole ? out + ((size_t)b * H_q + (size_t)h * G) * D : slot_ptr((int64_t)u + cta), sole);
        } else {
            if (last_seg) griddep_launch_dependents();
            griddep_wait();  // (early inputs) nothing is written before the wait
            if (sole) {  // no pages and no other partial: the output is zero
                float* o = out + ((size_t)b * H_q + (size_t)h * G) * D;
                for (int i = tid; i < G * D; i += NW * 32) o[i] = 0.f;
            } else {
                publish_slot<NW, MAXG>(sm.ms, sm.ms.o_final, G, slot_ptr((int64_t)u + cta), true);
            }
        }
        if (!sole) finish_unit(u);
        if constexpr (MODE == MODE_WINDOW) {
            if (pb == vmp) {  // CTA-uniform: this share holds the unit's last virtual page
                // The unit's BF16 window, attended exactly in the original
                // basis (the output basis), is one more partial of the unit:
                // published (even after a timed-out wait, so that the unit's
                // ticket completes) in slot units + n_cta + u.
                window_partials<NW, MAXG>(sm.o_part, sm.ms, q, H_q, H_kv, G, b, h, mu, win_k, win_v, win_lens,
                                          win_max, scale_log2);
                __syncthreads();
                merge_warps<NW, MAXG>(sm.ms, sm.o_part, G);
                publish_slot<NW, MAXG>(sm.ms, sm.ms.o_final, G, slot_ptr((int64_t)B * H_kv + n_cta + u), false);
                finish_unit(u);
            }
        }
        __syncthreads();  // the next segment reuses the ring and the merge scratch
    };
    segment(u_first, false);
    if (sm.share[1] > (int64_t)(u_first + 1) * vmp) segment(u_first + 1, true);
}

}  // namespace kvq

using namespace kvq;

// The dynamic shared memory opt-in is a per-device attribute of the kernel:
// set it on the first call on each device only.
static kvq_status set_smem_once(const void* fn, int bytes, int which) {
    static std::mutex mu;
    static bool done[64][6] = {};
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

// Streaming multiprocessors of the current device (looked up once per
// device); 152 (a GB300) where no device can be queried, so the host-only
// sizing helpers still answer on a machine without a GPU.
int kvq_device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

// Page CTAs of the INT2 decode: num_splits per (sequence, KV head) unit when
// given, else one wave (one CTA per SM) with at least 32 pages of the
// virtual page space per CTA; never fewer CTAs than units (so a CTA's share
// spans at most two units) and never more than virtual pages (so every share
// holds a page).  The count grows with the virtual pages per unit.
static int64_t int2_page_ctas(int B, int H_kv, int max_pages, int num_splits) {
    const int64_t units = (int64_t)B * H_kv, V = units * max_pages;
    int64_t C;
    if (num_splits > 0) {
        C = (int64_t)num_splits * units;
    } else {
        const int64_t nsm = kvq_device_sm_count();
        C = nsm;
        const int64_t cap = (V + 31) / 32;
        if (C > cap) C = cap;
        // a CTA's share must not span more than two units
        if (C < units) C = units;
    }
    if (C > V) C = V;
    return C;
}

// Virtual pages per unit of a decode step: in a decode step the CTA holding
// a sequence's new token also quantises and attends it (a few microseconds,
// about as long as streaming ~100 pages), so each unit gets that many
// virtual pages without work after its last page, and the share holding a
// full sequence's last page streams fewer real ones.  Below 96 pages a
// unit is one CTA's work anyway, and the extra pages would only add a
// second CTA (and a split-K merge) to it.
static int step_virtual_pages(int max_pages) { return max_pages + (max_pages < 96 ? 0 : 96); }

// Virtual pages per unit of a window decode: the CTA holding a unit's last
// virtual page attends its BF16 window after its pages, so each unit gets
// one page without work per window row (win_max, at most WIN_MAX_PAGES)
// after its last page.  The window's rows are read while the other CTAs
// still stream the cache, each request queued behind their copies, which
// makes a row cost about as much time as a page (measured: 33, 66, 132 and
// 264 such pages for a 132-row window at 128K gave the window 4.9, 4.1,
// 2.8 and 3.7 us over the plain decode).  Below 96 pages, as in the decode
// step, a unit is one CTA's work anyway.
constexpr int WIN_MAX_PAGES = 256;
static int window_virtual_pages(int max_pages, int win_max) {
    return max_pages + (max_pages < 96 ? 0 : win_max < WIN_MAX_PAGES ? win_max : WIN_MAX_PAGES);
}

extern "C" int kvq_decode_auto_splits(int B, int H_q, int H_kv, int max_pages_per_seq) {
    if (B <= 0 || H_kv <= 0 || H_q < H_kv || max_pages_per_seq <= 0) return 1;
    // at most one wave of CTAs, one per SM, over the (sequence, KV head)
    // pairs (a CTA past the wave would run alone in a second one); at least
    // 32 pages per split (the CTAs have 8-12 warps)
    const long units = (long)B * H_kv;
    long s = (long)kvq_device_sm_count() / units;
    long max_s = (max_pages_per_seq + 31) / 32;
    if (max_s > MAX_SPLITS) max_s = MAX_SPLITS;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    return (int)s;
}

// Partial slots the INT2 decode uses: one per (unit, page CTA) pair (units +
// C - 1 at most) and, with the window, one per unit.
static size_t int2_workspace_bytes(int B, int H_q, int H_kv, int64_t slots) {
    const int G = (H_q + H_kv - 1) / H_kv;
    return WS_HEADER + tickets_bytes(B, H_kv) + (size_t)slots * G * PART_STRIDE * sizeof(float);
}

extern "C" size_t kvq_decode_workspace_bytes(int B, int H_q, int H_kv, int max_pages_per_seq, int num_splits) {
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || max_pages_per_seq <= 0 || max_pages_per_seq > (1 << 28) ||
        num_splits < 0)
        return 0;
    const int64_t units = (int64_t)B * H_kv;
    int64_t slots;
    if (num_splits > 0) {
        // INT2 with and without the window, and Block-GTQ's num_splits per unit
        slots = ((int64_t)num_splits + 2) * units;
    } else {  // room for the automatic choice of every decode entry point
        const int64_t plain = units + int2_page_ctas(B, H_kv, max_pages_per_seq, 0);
        const int64_t step = units + int2_page_ctas(B, H_kv, step_virtual_pages(max_pages_per_seq), 0);
        // the window's pages without work are at most WIN_MAX_PAGES per unit
        const int64_t win = 2 * units + int2_page_ctas(B, H_kv, window_virtual_pages(max_pages_per_seq, 1 << 30), 0);
        const int64_t bg = units * bgtq_decode_auto_splits(B, H_q, H_kv, max_pages_per_seq);
        slots = plain > win ? plain : win;
        if (step > slots) slots = step;
        if (bg > slots) slots = bg;
    }
    return int2_workspace_bytes(B, H_q, H_kv, slots);
}

// Test hook: makes the next INT2 decode launch on this process drop one bulk
// copy so that a bounded wait runs out (kvq_debug_drop_next_copy).
static std::atomic<int> g_debug_flags{0};

extern "C" void kvq_debug_drop_next_copy(void) { g_debug_flags.store(DBG_DROP_FIRST_COPY); }

// A validated INT2 decode launch.
struct Int2Plan {
    int G = 0, C = 0, grid = 0, threads = 0, mode = MODE_CACHE, vmp = 0;
    size_t smem = 0, need = 0;
};

// Argument checks shared by the INT2 decode entry points (nothing is
// enqueued).  mode MODE_WINDOW: win_k, win_v, win_lens, win_max and mu_k
// describe the BF16 window; MODE_STEP: win_k, win_v are the new token's key
// and value and mu_k the key centre.  workspace is checked for null and
// alignment only when check_ws is set.
static kvq_status decode_int2_plan(const char* fn, int mode, const void* q, int B, int H_q, int H_kv, int d,
                                   const void* cache, int64_t num_pages, const int32_t* block_table,
                                   int max_pages_per_seq, const int32_t* context_lens, const float* R_k,
                                   const float* R_v, const float* mu_k, const void* win_k, const void* win_v,
                                   const int32_t* win_lens, int win_max, float* out, const void* workspace,
                                   bool check_ws, int num_splits, Int2Plan& plan) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: d=%d (only 128)", fn, d);
    if (B <= 0 || H_kv <= 0 || H_q <= 0 || H_q % H_kv || max_pages_per_seq <= 0 || num_pages <= 0 ||
        num_splits < 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: B=%d H_q=%d H_kv=%d max_pages=%d num_pages=%lld splits=%d",
                             fn, B, H_q, H_kv, max_pages_per_seq, (long long)num_pages, num_splits);
    const int G = H_q / H_kv;
    if (G > 8) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: GQA group %d > 8", fn, G);
    if (B > 65535 || H_kv > 65535) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: B or H_kv above 65535", fn);
    if ((int64_t)B * H_kv * max_pages_per_seq > (int64_t(1) << 40))
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: B * H_kv * max_pages above 2^40", fn);
    // (an int32 context spans at most 2^27 pages; the bound keeps the virtual
    // pages per unit, max_pages plus a few hundred, within int)
    if (max_pages_per_seq > (1 << 28))
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: max_pages_per_seq %d above 2^28", fn, max_pages_per_seq);
    if (num_splits > MAX_SPLITS - 2)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: %d splits above %d", fn, num_splits, MAX_SPLITS - 2);
    if (!q || !cache || !block_table || !context_lens || !R_k || !R_v || !out || (check_ws && !workspace))
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (reinterpret_cast<uintptr_t>(cache) % 16 || (check_ws && reinterpret_cast<uintptr_t>(workspace) % 16) ||
        reinterpret_cast<uintptr_t>(R_k) % 16 || reinterpret_cast<uintptr_t>(R_v) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: cache, R_k, R_v and workspace need 16-byte alignment", fn);
    if (mode == MODE_WINDOW) {
        if (!win_k || win_max <= 0 || !win_v || !win_lens || !mu_k)
            return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: window needs win_max > 0, win_v, win_lens and mu_k", fn);
        if (reinterpret_cast<uintptr_t>(win_k) % 16 || reinterpret_cast<uintptr_t>(win_v) % 16)
            return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: win_k and win_v need 16-byte alignment", fn);
    }
    if (mode == MODE_STEP && (!win_k || !win_v || !mu_k))
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: null k_new, v_new or mu_k", fn);
    const bool win = mode == MODE_WINDOW;  // one window partial per unit
    const int64_t units = (int64_t)B * H_kv;
    const int vmp = mode == MODE_STEP     ? step_virtual_pages(max_pages_per_seq)
                    : mode == MODE_WINDOW ? window_virtual_pages(max_pages_per_seq, win_max)
                                          : max_pages_per_seq;
    if ((int64_t)B * H_kv * vmp > (int64_t(1) << 40))
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: B * H_kv * max_pages above 2^40", fn);
    const int64_t C = int2_page_ctas(B, H_kv, vmp, num_splits);
    // a unit's partials: the page CTAs over its pages (its share of the
    // virtual pages spans at most ceil(C / units) + 1 of them) and the window
    if ((C + units - 1) / units + 2 > MAX_SPLITS)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "%s: %lld CTAs over %lld units exceed %d partials per unit", fn,
                             (long long)C, (long long)units, MAX_SPLITS);
    if (C > 0x7fffffff) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "%s: grid of %lld CTAs", fn, (long long)C);
    constexpr int NW1 = DecWarps<1>::NW, NW2 = DecWarps<2>::NW;
    plan.G = G;
    plan.C = (int)C;
    plan.grid = (int)C;
    plan.mode = mode;
    plan.vmp = vmp;
    plan.threads = (G <= 4 ? NW1 : NW2) * 32;
    plan.smem = G <= 4 ? sizeof(DecodeSmem<NW1, 4>) : sizeof(DecodeSmem<NW2, 8>);
    plan.need = int2_workspace_bytes(B, H_q, H_kv, units + C + (win ? units : 0));
    return KVQ_OK;
}

static kvq_status decode_int2_launch(const Int2Plan& plan, const void* q, int B, int H_q, int H_kv,
                                     void* cache, int64_t num_pages, const int32_t* block_table,
                                     int max_pages_per_seq, const int32_t* context_lens, const float* R_k,
                                     const float* R_v, const float* mu_k, const void* win_k, const void* win_v,
                                     const int32_t* win_lens, int win_max, float scale, float* out, void* workspace,
                                     void* stream, int kernel_flags = 0) {
    const float scale_log2 = scale * 1.4426950408889634f;
    const bool small = plan.G <= 4;
    using Kern = decltype(&decode_int2_kernel<1, MODE_CACHE>);
    static const Kern kerns[2][3] = {
        {decode_int2_kernel<1, MODE_CACHE>, decode_int2_kernel<1, MODE_WINDOW>, decode_int2_kernel<1, MODE_STEP>},
        {decode_int2_kernel<2, MODE_CACHE>, decode_int2_kernel<2, MODE_WINDOW>, decode_int2_kernel<2, MODE_STEP>}};
    const Kern kern = kerns[small ? 0 : 1][plan.mode];
    kvq_status sa = set_smem_once((const void*)kern, (int)plan.smem, (small ? 0 : 3) + plan.mode);
    if (sa != KVQ_OK) return sa;
    const int flags = g_debug_flags.exchange(0) | kernel_flags;
    const cudaError_t e = launch_pdl(
        kern, dim3(plan.grid), dim3(plan.threads), plan.smem, static_cast<cudaStream_t>(stream),
        static_cast<const __nv_bfloat16*>(q), B, H_q, H_kv, plan.G, static_cast<uint8_t*>(cache), num_pages,
        block_table, max_pages_per_seq, context_lens, R_k, R_v, mu_k, static_cast<const __nv_bfloat16*>(win_k),
        static_cast<const __nv_bfloat16*>(win_v), win_lens, win_max, scale_log2, out,
        static_cast<uint8_t*>(workspace), plan.C, plan.vmp, flags);
    return kvq_check_cuda(e, "decode launch");
}

extern "C" kvq_status kvq_decode_attn_int2(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                           int64_t num_pages, const int32_t* block_table, int max_pages_per_seq,
                                           const int32_t* context_lens, const float* R_k, const float* R_v,
                                           float scale, float* out, void* workspace, size_t workspace_bytes,
                                           int num_splits, void* stream) {
    Int2Plan plan;
    kvq_status st = decode_int2_plan("kvq_decode_attn_int2", MODE_CACHE, q, B, H_q, H_kv, d, cache, num_pages, block_table,
                                     max_pages_per_seq, context_lens, R_k, R_v, nullptr, nullptr, nullptr, nullptr,
                                     0, out, workspace, true, num_splits, plan);
    if (st != KVQ_OK) return st;
    if (workspace_bytes < plan.need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "kvq_decode_attn_int2: workspace %zu < %zu bytes", workspace_bytes,
                             plan.need);
    return decode_int2_launch(plan, q, B, H_q, H_kv, const_cast<void*>(cache), num_pages, block_table,
                              max_pages_per_seq, context_lens, R_k, R_v, nullptr, nullptr, nullptr, nullptr, 0, scale,
                              out, workspace, stream);
}

extern "C" kvq_status kvq_decode_attn_int2_window(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                                  int64_t num_pages, const int32_t* block_table,
                                                  int max_pages_per_seq, const int32_t* context_lens,
                                                  const float* R_k, const float* R_v, const float* mu_k,
                                                  const void* win_k, const void* win_v, const int32_t* win_lens,
                                                  int win_max, float scale, float* out, void* workspace,
                                                  size_t workspace_bytes, int num_splits, void* stream) {
    if (!win_k) return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_decode_attn_int2_window: null win_k");
    Int2Plan plan;
    kvq_status st = decode_int2_plan("kvq_decode_attn_int2_window", MODE_WINDOW, q, B, H_q, H_kv, d, cache, num_pages,
                                     block_table, max_pages_per_seq, context_lens, R_k, R_v, mu_k, win_k, win_v,
                                     win_lens, win_max, out, workspace, true, num_splits, plan);
    if (st != KVQ_OK) return st;
    if (workspace_bytes < plan.need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "kvq_decode_attn_int2_window: workspace %zu < %zu bytes",
                             workspace_bytes, plan.need);
    return decode_int2_launch(plan, q, B, H_q, H_kv, const_cast<void*>(cache), num_pages, block_table,
                              max_pages_per_seq, context_lens, R_k, R_v, mu_k, win_k, win_v, win_lens, win_max, scale,
                              out, workspace, stream);
}

extern "C" kvq_status kvq_decode_step_int2(const void* q, const void* k_new, const void* v_new, int B, int H_q,
                                           int H_kv, int d, void* cache, int64_t num_pages,
                                           const int32_t* block_table, int max_pages_per_seq,
                                           const int32_t* context_lens, const float* mu_k, const float* R_k,
                                           const float* R_v, float scale, float* out, void* workspace,
                                           size_t workspace_bytes, int num_splits, int flags, void* stream) {
    if (flags & ~KVQ_STEP_INPUTS_READY)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_decode_step_int2: unknown flags %d", flags);
    Int2Plan plan;
    kvq_status st = decode_int2_plan("kvq_decode_step_int2", MODE_STEP, q, B, H_q, H_kv, d, cache, num_pages,
                                     block_table, max_pages_per_seq, context_lens, R_k, R_v, mu_k, k_new, v_new,
                                     nullptr, 0, out, workspace, true, num_splits, plan);
    if (st != KVQ_OK) return st;
    if (workspace_bytes < plan.need)
        return kvq_set_error(KVQ_ERR_WORKSPACE, "kvq_decode_step_int2: workspace %zu < %zu bytes", workspace_bytes,
                             plan.need);
    return decode_int2_launch(plan, q, B, H_q, H_kv, cache, num_pages, block_table, max_pages_per_seq, context_lens,
                              R_k, R_v, mu_k, k_new, v_new, nullptr, 0, scale, out, workspace, stream,
                              (flags & KVQ_STEP_INPUTS_READY) ? FLAG_EARLY_INPUTS : 0);
}

// Checks and launch used by kvq_decode_attn_int2_noalloc (its own file): the
// arguments are validated before `prepare` runs, which may enqueue work on
// the scratch it returns.
kvq_status kvq_decode_int2_checked(const char* fn, const void* q, int B, int H_q, int H_kv, int d,
                                   const void* cache, int64_t num_pages, const int32_t* block_table,
                                   int max_pages_per_seq, const int32_t* context_lens, const float* R_k,
                                   const float* R_v, float scale, float* out, int num_splits, void* stream,
                                   size_t scratch_bytes, kvq_status (*prepare)(size_t zeroed, void* stream, void** ws)) {
    Int2Plan plan;
    kvq_status st = decode_int2_plan(fn, MODE_CACHE, q, B, H_q, H_kv, d, cache, num_pages, block_table, max_pages_per_seq,
                                     context_lens, R_k, R_v, nullptr, nullptr, nullptr, nullptr, 0, out, nullptr,
                                     false, num_splits, plan);
    if (st != KVQ_OK) return st;
    if (plan.need > scratch_bytes)
        return kvq_set_error(KVQ_ERR_WORKSPACE,
                             "%s: this shape needs %zu bytes of scratch, above the fixed %zu; use "
                             "kvq_decode_attn_int2 with a workspace, or fewer splits",
                             fn, plan.need, scratch_bytes);
    void* ws = nullptr;
    st = prepare(WS_HEADER + tickets_bytes(B, H_kv), stream, &ws);
    if (st != KVQ_OK) return st;
    return decode_int2_launch(plan, q, B, H_q, H_kv, const_cast<void*>(cache), num_pages, block_table,
                              max_pages_per_seq, context_lens, R_k, R_v, nullptr, nullptr, nullptr, nullptr, 0, scale,
                              out, ws, stream);
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
