// Shared device helpers for the rotated low-bit KV-cache kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int D = 128;          // head dimension
constexpr int PAGE = 16;        // tokens per page
constexpr int NGROUP = 4;       // INT2 groups of 32 channels

// INT2 tile of one (page, KV head)
constexpr int INT2_TILE = 1536;
constexpr int OFF_KC = 0, OFF_KM = 512, OFF_VC = 768, OFF_VM = 1280;
// Key meta: per slot 16 bytes, one (fp16 scale, fp16 min) word per group.
// Value meta: pair-major, so a word holds one group's scales (or mins) of
// slots 2j and 2j + 1 -- the order the PV step multiplies them in:
// scales at OFF_VM + 16 j + 4 g (+2 for the odd slot), mins VM_MINS later.
constexpr int VM_MINS = 128;
__host__ __device__ constexpr int vm_scale_off(int s, int g) { return OFF_VM + 16 * (s >> 1) + 4 * g + 2 * (s & 1); }

// decode workspace: [header 256 B][tickets][partials]
constexpr int WS_HEADER = 256;
constexpr int PART_STRIDE = 132;  // floats per (seq, q head, split): m, l, pad, pad, o[128]
constexpr uint32_t ERR_BAD_PAGE = 1u, ERR_TIMEOUT = 2u, ERR_BAD_WIDTHS = 4u;

// give an mbarrier wait about two seconds at ~2 GHz before declaring failure
constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// one int32 split ticket per (sequence, KV head), zero between calls
__host__ __device__ inline size_t tickets_bytes(int B, int H_kv) { return align_up((size_t)B * H_kv * 4, 256); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace kvq

// Automatic split count of the Block-GTQ decode (host).
int bgtq_decode_auto_splits(int B, int H_q, int H_kv, int max_pages_per_seq);

// Streaming multiprocessors of the current device (host; 152 without one).
int kvq_device_sm_count();

// The INT2 decode with every argument validated before `prepare` is called
// to clear (`zeroed` bytes) and return the scratch it runs in (host; used by
// the allocation-free entry point).
kvq_status kvq_decode_int2_checked(const char* fn, const void* q, int B, int H_q, int H_kv, int d,
                                   const void* cache, int64_t num_pages, const int32_t* block_table,
                                   int max_pages_per_seq, const int32_t* context_lens, const float* R_k,
                                   const float* R_v, float scale, float* out, int num_splits, void* stream,
                                   size_t scratch_bytes, kvq_status (*prepare)(size_t zeroed, void* stream, void** ws));

namespace kvq {

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for an mbarrier phase with a time limit; false when the limit passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}

// atomicAdd at GPU scope with acquire-release order: writes ordered before it
// (in the CTA, by a preceding __syncthreads) are visible to any thread that
// acquires the value it leaves, and reads ordered after it see what the
// earlier adders released.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization (launch_pdl): it may be scheduled
// while the kernel before it in the stream is still finishing, so it calls
// griddep_wait() before its first read of global memory that kernel may have
// written (a no-op when launched without the attribute), and calls
// griddep_launch_dependents() once the kernel after it may be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Ask L2 to fetch the 128-byte line at p and keep it ahead of streaming data.
// Fetch a line into L2 without returning data.  L2 is the point of
// coherence for global memory, so a prefetch issued before
// griddepcontrol.wait cannot hand a later load a stale value: a write the
// previous kernel makes afterwards lands in L2 too.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

// 1-D bulk copy global -> shared (16-byte aligned, size multiple of 16),
// completion signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// An L2 policy that marks lines evict-first: for data streamed once, so it
// does not push out of L2 what is read again (code, rotations, queries,
// block tables).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy (l2_policy_evict_first for a stream).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Error-free sum: a + b == s + e exactly (no contraction, fixed rounding).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// x - m > t exactly, given fp32 x, m and an exactly representable fp32 t.
__device__ __forceinline__ bool diff_gt(float hi, float lo, float t) { return hi > t || (hi == t && lo > 0.f); }

// fp32 -> fp16 round-to-nearest-even, saturating at +-65504.
__device__ __forceinline__ __half f16_sat(float x) {
    return __float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f));
}

}  // namespace kvq

// thread-local error text lives in host.cpp
kvq_status kvq_set_error(kvq_status st, const char* fmt, ...);
kvq_status kvq_check_cuda(cudaError_t e, const char* what);
