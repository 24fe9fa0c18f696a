// Quantise-on-append for the rotated INT2 KV cache.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization": the key is centred
// (§1, attention-equivalent reparameterisation) and rotated, z = (k - mu) R_k;
// the value is rotated, w = v R_v (§3.1 Eq. 4); each group of 32 rotated
// channels is INT2-quantised with one fp16 scale and min (§1).
//
// One CTA = 64 threads works on one (KV head, 32-channel group) and a run of
// tokens.  Warp 0 produces the group's 32 rotated key channels, warp 1 the
// group's 32 rotated value channels; each thread keeps its column of the
// rotation in registers, so R is read once per CTA and a single appended
// token is spread over 4 CTAs per head.  A rotated coordinate is a
// fixed-order fp32 fma chain over the 128 inputs (the order the format's
// documentation promises).  Within the warp: min/max by shuffles, exact
// threshold comparisons, and the four 2-bit codes of a byte gathered from
// four neighbouring lanes.  Appends of 256 tokens or more (prefill) take a
// register-tiled kernel with R in shared memory that runs the same chains.
#include <mutex>

#include "int2_quant.cuh"

namespace kvq {

__global__ void __launch_bounds__(64)
append_int2_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, int n_tok,
                   int H_kv, const int32_t* __restrict__ slot_mapping, const float* __restrict__ mu,
                   const float* __restrict__ Rk, const float* __restrict__ Rv, uint8_t* __restrict__ cache,
                   int64_t num_pages, float* __restrict__ dbg_k, float* __restrict__ dbg_v,
                   int32_t* __restrict__ err_count, int tok_per_cta, float clip) {
    griddep_launch_dependents();
    const int h = blockIdx.y, grp = blockIdx.z;
    const int tid = threadIdx.x;
    const int is_v = tid >> 5;
    const int lane = tid & 31;
    const int j = 32 * grp + lane;  // output channel

    // this thread's column of the rotation: its 128-byte row segments are
    // fetched into L2 while the previous kernel in the stream may still be
    // running (a prefetch returns no data; L2 is the point of coherence, so
    // a later write by that kernel still wins), and read after the wait
    const float* R = (is_v ? Rv : Rk) + (size_t)h * D * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) prefetch_l2(R + (size_t)(lane + 32 * e) * D + 32 * grp);
    griddep_wait();  // every input (rotations included) may come from the previous kernel
    float rcol[D];
#pragma unroll
    for (int i = 0; i < D; ++i) rcol[i] = __ldg(R + i * D + j);

    __shared__ float xs[2][2][D];
    const int t0 = blockIdx.x * tok_per_cta;
    const int t1 = min(n_tok, t0 + tok_per_cta);
    const int64_t n_slots = num_pages * PAGE;
    int buf = 0;

    for (int t = t0; t < t1; ++t) {
        const int slot = __ldg(slot_mapping + t);
        if (slot < 0 && slot != -1) {
            if (tid == 0 && h == 0 && grp == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        if (slot == -1) continue;
        if ((int64_t)slot >= n_slots) {
            if (tid == 0 && h == 0 && grp == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        // stage the token's key (centred) and value rows: 4 + 4 inputs per thread
        {
            const __nv_bfloat16* src = (is_v ? v : k) + ((size_t)t * H_kv + h) * D;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = lane + 32 * e;
                float x = __bfloat162float(src[i]);
                if (!is_v) x = __fsub_rn(x, __ldg(mu + h * D + i));
                xs[buf][is_v][i] = x;
            }
        }
        __syncthreads();

        const float* xv = xs[buf][is_v];
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < D; ++i) acc = __fmaf_rn(xv[i], rcol[i], acc);
        buf ^= 1;

        float* dbg = is_v ? dbg_v : dbg_k;
        if (dbg) dbg[((size_t)t * H_kv + h) * D + j] = acc;

        // group parameters (exact min / max over the 32 lanes)
        float mn = acc, mx = acc;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        __half sh, mh;
        int2_params(mn, mx, clip, sh, mh);
        const int code = int2_code(acc, __half2float(mh), __half2float(sh));

        // byte 4*b + g holds channels 32g + 4b + c at bits 2c
        uint32_t bits = (uint32_t)code << (2 * (lane & 3));
        bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
        const int page = slot / PAGE, s = slot % PAGE;
        uint8_t* tile = cache + ((size_t)page * H_kv + h) * INT2_TILE;
        uint8_t* rec = tile + (is_v ? OFF_VC : OFF_KC) + 32 * s;
        if ((lane & 3) == 0) rec[4 * (lane >> 2) + grp] = (uint8_t)bits;
        if (lane == 0) int2_store_meta(tile, is_v, s, grp, sh, mh);
    }
}

// Prefill-sized appends: the same chains, register-tiled.  A CTA of 256
// threads takes one (KV head, side) and PF_TILES tiles of PF_TOK tokens;
// R (64 KB) is staged in shared memory once, each tile's inputs are stored
// transposed (X[i][token]).  Thread (warp w, lane l) owns channels
// 4l .. 4l+3 -- one byte of the code record (group l / 8, byte-row l % 8)
// -- for tokens 8w .. 8w+7 of the tile: per input index i it reads R[i][4l
// .. 4l+3] and X[i][8w .. 8w+7] and runs 32 chains one step, each chain the
// same fixed-order fp32 fma sequence over i = 0 .. 127 as above, so the
// codes are the same bit for bit.  A group's 32 channels sit in 8
// neighbouring lanes (min / max over 3 shuffles), and a warp writes whole
// 32-byte code records.
constexpr int PF_TOK = 64;
constexpr int PF_TILES = 4;
constexpr int PF_XS = PF_TOK + 4;  // padded transposed-tile row (16-byte multiple)

struct __align__(16) PrefillSmem {
    float R[D][D];
    float X[D][PF_XS];
    int slot[PF_TOK];
};

__global__ void __launch_bounds__(256, 2)
append_int2_prefill_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, int n_tok,
                           int H_kv, const int32_t* __restrict__ slot_mapping, const float* __restrict__ mu,
                           const float* __restrict__ Rk, const float* __restrict__ Rv, uint8_t* __restrict__ cache,
                           int64_t num_pages, float* __restrict__ dbg_k, float* __restrict__ dbg_v,
                           int32_t* __restrict__ err_count, float clip) {
    griddep_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);
    const int h = blockIdx.y, is_v = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    {
        // the rotation: fetched into L2 before the dependency wait (no data
        // returned, coherent), staged in shared memory after it
        const float4* R4 = reinterpret_cast<const float4*>((is_v ? Rv : Rk) + (size_t)h * D * D);
        for (int l = tid; l < D * D * 4 / 128; l += 256) prefetch_l2(R4 + 8 * l);
        griddep_wait();  // every input (rotations included) may come from the previous kernel
        float4* S4 = reinterpret_cast<float4*>(&sm.R[0][0]);
        for (int idx = tid; idx < D * D / 4; idx += 256) S4[idx] = __ldg(R4 + idx);
    }

    const __nv_bfloat16* src = is_v ? v : k;
    const int64_t n_slots = num_pages * PAGE;
    const int g = lane >> 3, row = lane & 7;  // this lane's group and byte-row
    float* dbg = is_v ? dbg_v : dbg_k;
    // a tile's inputs: job (half, chunk) of this warp = tokens t0 + 32 half +
    // lane, channels 8 chunk .. +7; loaded into registers one tile ahead
    uint4 raw[4];
    int slot_pf = -1;
    auto load_tile = [&](int t0) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int job = warp + 8 * m, half = job >> 4, c = job & 15, t = t0 + 32 * half + lane;
            raw[m] = t < n_tok ? __ldg(reinterpret_cast<const uint4*>(src + ((size_t)t * H_kv + h) * D + 8 * c))
                               : make_uint4(0u, 0u, 0u, 0u);
        }
        slot_pf = tid < PF_TOK && t0 + tid < n_tok ? __ldg(slot_mapping + t0 + tid) : -1;
    };
    const int tile0 = blockIdx.x * PF_TILES * PF_TOK;
    if (tile0 < n_tok) load_tile(tile0);
    for (int tl = 0; tl < PF_TILES; ++tl) {
        const int t0 = tile0 + tl * PF_TOK;
        if (t0 >= n_tok) break;
        __syncthreads();  // the previous tile's inputs are consumed
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int job = warp + 8 * m, half = job >> 4, c = job & 15, tt = 32 * half + lane;
            const uint32_t w[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
            float x[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = __uint_as_float(w[e] << 16);
                x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
            if (!is_v && t0 + tt < n_tok) {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __fsub_rn(x[e], __ldg(mu + h * D + 8 * c + e));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sm.X[8 * c + e][tt] = x[e];
        }
        if (tid < PF_TOK) sm.slot[tid] = slot_pf;
        __syncthreads();
        if (tl + 1 < PF_TILES && t0 + PF_TOK < n_tok) load_tile(t0 + PF_TOK);

        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[a][u] = 0.f;
#pragma unroll 4
        for (int i = 0; i < D; ++i) {
            const float4 r4 = *reinterpret_cast<const float4*>(&sm.R[i][4 * lane]);
            const float4 xa = *reinterpret_cast<const float4*>(&sm.X[i][8 * warp]);
            const float4 xb = *reinterpret_cast<const float4*>(&sm.X[i][8 * warp + 4]);
            const float rc[4] = {r4.x, r4.y, r4.z, r4.w};
            const float xt[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[a][u] = __fmaf_rn(xt[u], rc[a], acc[a][u]);
        }

#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int tt = 8 * warp + u, t = t0 + tt;
            if (t >= n_tok) break;               // warp-uniform
            const int slot = sm.slot[tt];        // warp-uniform
            if (slot == -1) continue;
            if (slot < -1 || (int64_t)slot >= n_slots) {
                if (lane == 0 && h == 0 && is_v == 0 && err_count) atomicAdd(err_count, 1);
                continue;
            }
            if (dbg)
                *reinterpret_cast<float4*>(dbg + ((size_t)t * H_kv + h) * D + 4 * lane) =
                    make_float4(acc[0][u], acc[1][u], acc[2][u], acc[3][u]);
            float mn = fminf(fminf(acc[0][u], acc[1][u]), fminf(acc[2][u], acc[3][u]));
            float mx = fmaxf(fmaxf(acc[0][u], acc[1][u]), fmaxf(acc[2][u], acc[3][u]));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            __half sh, mh;
            int2_params(mn, mx, clip, sh, mh);
            const float scf = __half2float(sh), mnf = __half2float(mh);
            uint32_t byte = 0;
#pragma unroll
            for (int a = 0; a < 4; ++a) byte |= (uint32_t)int2_code(acc[a][u], mnf, scf) << (2 * a);
            const int page = slot / PAGE, s = slot % PAGE;
            uint8_t* tile = cache + ((size_t)page * H_kv + h) * INT2_TILE;
            // channels 32g + 4 row + a sit in byte 4 row + g, bits 2a
            tile[(is_v ? OFF_VC : OFF_KC) + 32 * s + 4 * row + g] = (uint8_t)byte;
            if (row == 0) int2_store_meta(tile, is_v, s, g, sh, mh);
        }
    }
}

}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_int2_tile_bytes(int d) { return d == D ? (size_t)INT2_TILE : 0; }

// appends of at least this many tokens take the register-tiled kernel
static constexpr int PREFILL_MIN_TOKENS = 256;

static kvq_status append_int2_launch(const void* k, const void* v, int n_tok, int H_kv, int d,
                                      const int32_t* slot_mapping, const float* mu_k, const float* R_k,
                                      const float* R_v, void* cache, int64_t num_pages, float* dbg_rot_k,
                                      float* dbg_rot_v, int32_t* err_count, float clip, void* stream) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "kvq_append_int2: d=%d (only 128)", d);
    if (n_tok < 0 || H_kv <= 0 || num_pages <= 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_append_int2: n_tok=%d H_kv=%d num_pages=%lld", n_tok,
                             H_kv, (long long)num_pages);
    if (H_kv > 65535) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "kvq_append_int2: H_kv=%d too large", H_kv);
    if (!(clip > 0.f && clip <= 1.f))
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_append_int2: clip ratio %g outside (0, 1]", (double)clip);
    if (n_tok == 0) return KVQ_OK;
    if (!k || !v || !slot_mapping || !mu_k || !R_k || !R_v || !cache)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_append_int2: null pointer");
    if (reinterpret_cast<uintptr_t>(cache) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_append_int2: cache not 16-byte aligned");

    const bool aligned = reinterpret_cast<uintptr_t>(k) % 16 == 0 && reinterpret_cast<uintptr_t>(v) % 16 == 0 &&
                         (!dbg_rot_k || reinterpret_cast<uintptr_t>(dbg_rot_k) % 16 == 0) &&
                         (!dbg_rot_v || reinterpret_cast<uintptr_t>(dbg_rot_v) % 16 == 0);
    if (n_tok >= PREFILL_MIN_TOKENS && aligned) {
        // prefill: the register-tiled kernel (same arithmetic, same codes)
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        kvq_status s2 = kvq_check_cuda(cudaGetDevice(&dev), "kvq_append_int2: cudaGetDevice");
        if (s2 != KVQ_OK) return s2;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (dev < 0 || dev >= 64 || !done[dev]) {
                s2 = kvq_check_cuda(cudaFuncSetAttribute((const void*)append_int2_prefill_kernel,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)sizeof(PrefillSmem)),
                                    "kvq_append_int2 smem attribute");
                if (s2 != KVQ_OK) return s2;
                if (dev >= 0 && dev < 64) done[dev] = true;
            }
        }
        const int per_cta = PF_TOK * PF_TILES;
        dim3 grid((n_tok + per_cta - 1) / per_cta, H_kv, 2);
        return kvq_check_cuda(
            launch_pdl(append_int2_prefill_kernel, grid, dim3(256), sizeof(PrefillSmem), static_cast<cudaStream_t>(stream),
                       static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), n_tok, H_kv,
                       slot_mapping, mu_k, R_k, R_v, static_cast<uint8_t*>(cache), num_pages, dbg_rot_k, dbg_rot_v,
                       err_count, clip),
            "kvq_append_int2 launch");
    }
    // enough CTAs for about four waves of the 152 SMs; at most 64 tokens each
    const int want_ctas = 152 * 16;
    int chunks = (want_ctas + 4 * H_kv - 1) / (4 * H_kv);
    chunks = chunks < 1 ? 1 : chunks;
    int per = (n_tok + chunks - 1) / chunks;
    per = per < 1 ? 1 : (per > 64 ? 64 : per);
    const int grid_x = (n_tok + per - 1) / per;
    dim3 grid(grid_x, H_kv, NGROUP);
    return kvq_check_cuda(launch_pdl(append_int2_kernel, grid, dim3(64), 0, static_cast<cudaStream_t>(stream),
                                     static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), n_tok,
                                     H_kv, slot_mapping, mu_k, R_k, R_v, static_cast<uint8_t*>(cache), num_pages,
                                     dbg_rot_k, dbg_rot_v, err_count, per, clip),
                          "kvq_append_int2 launch");
}

extern "C" kvq_status kvq_append_int2(const void* k, const void* v, int n_tok, int H_kv, int d,
                                      const int32_t* slot_mapping, const float* mu_k, const float* R_k,
                                      const float* R_v, void* cache, int64_t num_pages, float* dbg_rot_k,
                                      float* dbg_rot_v, int32_t* err_count, void* stream) {
    return append_int2_launch(k, v, n_tok, H_kv, d, slot_mapping, mu_k, R_k, R_v, cache, num_pages, dbg_rot_k,
                              dbg_rot_v, err_count, 1.0f, stream);
}

extern "C" kvq_status kvq_append_int2_clip(const void* k, const void* v, int n_tok, int H_kv, int d,
                                           const int32_t* slot_mapping, const float* mu_k, const float* R_k,
                                           const float* R_v, float clip, void* cache, int64_t num_pages,
                                           float* dbg_rot_k, float* dbg_rot_v, int32_t* err_count, void* stream) {
    return append_int2_launch(k, v, n_tok, H_kv, d, slot_mapping, mu_k, R_k, R_v, cache, num_pages, dbg_rot_k,
                              dbg_rot_v, err_count, clip, stream);
}

namespace kvq {

// Reads cached tokens back: thread (token, head, side, channel) forms
// min + code * scale with one fp32 fused multiply-add.
__global__ void __launch_bounds__(256)
dequant_int2_kernel(const uint8_t* __restrict__ cache, int64_t num_pages, int H_kv,
                    const int32_t* __restrict__ slot_mapping, int n, float* __restrict__ k_rot,
                    float* __restrict__ v_rot) {
    griddep_wait();
    griddep_launch_dependents();
    const int t = blockIdx.x, h = blockIdx.y;
    const int side = threadIdx.x >> 7, j = threadIdx.x & (D - 1);
    float* dst = side ? v_rot : k_rot;
    if (!dst) return;
    const int slot = __ldg(slot_mapping + t);
    float val = 0.f;
    if (slot >= 0 && (int64_t)slot < num_pages * PAGE) {
        const int page = slot / PAGE, s = slot % PAGE;
        const uint8_t* tile = cache + ((size_t)page * H_kv + h) * INT2_TILE;
        // channel j = 32 g + 4 b + c sits in byte 4 b + g, bits 2c
        const int g = j >> 5, b = (j >> 2) & 7, c = j & 3;
        const int code = (tile[(side ? OFF_VC : OFF_KC) + 32 * s + 4 * b + g] >> (2 * c)) & 3;
        const uint8_t* m = side ? tile + vm_scale_off(s, g) : tile + OFF_KM + 16 * s + 4 * g;
        const float sc = __half2float(*reinterpret_cast<const __half*>(m));
        const float mn = __half2float(*reinterpret_cast<const __half*>(m + (side ? VM_MINS : 2)));
        val = __fmaf_rn((float)code, sc, mn);
    }
    dst[((size_t)t * H_kv + h) * D + j] = val;
}

}  // namespace kvq

extern "C" kvq_status kvq_dequant_int2(const void* cache, int64_t num_pages, int H_kv, int d,
                                       const int32_t* slot_mapping, int n, float* k_rot, float* v_rot,
                                       void* stream) {
    if (d != D) return kvq_set_error(KVQ_ERR_UNSUPPORTED, "kvq_dequant_int2: d=%d (only 128)", d);
    if (n < 0 || H_kv <= 0 || H_kv > 65535 || num_pages <= 0 || n > 0x7fffffff)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_dequant_int2: n=%d H_kv=%d num_pages=%lld", n, H_kv,
                             (long long)num_pages);
    if (n == 0) return KVQ_OK;
    if (!cache || !slot_mapping || (!k_rot && !v_rot))
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_dequant_int2: null pointer");
    if (reinterpret_cast<uintptr_t>(cache) % 16)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "kvq_dequant_int2: cache not 16-byte aligned");
    return kvq_check_cuda(launch_pdl(dequant_int2_kernel, dim3(n, H_kv), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(cache),
                                     num_pages, H_kv, slot_mapping, n, k_rot, v_rot),
                          "kvq_dequant_int2 launch");
}
