// INT2 decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attn_int2 needs a caller-provided workspace for its split-K
// partials and tickets.  Some callers cannot produce one at call time: a
// serving loop whose device memory is planned once up front, a host that
// owns all device memory through its own allocator, or code where the
// device-wide synchronisation cudaMalloc may imply is not acceptable.  This
// entry point runs the same decode with its scratch in a fixed-size array
// that lives in the library's own device memory instead.
#include <mutex>

#include "kvq_common.cuh"

// 4 MiB of decode scratch, resident on every GPU that loads the library
// until the process exits.  All calls share it.
static constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_decode_scratch[kNoallocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  The name is
// only a host-side stand-in; the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current (so the entry point
// must not be used across a cudaDeviceReset, which may move the array).
kvq_status scratch_address(void** out) {
    int dev = 0;
    kvq_status st = kvq_check_cuda(cudaGetDevice(&dev), "kvq_decode_attn_int2_noalloc: cudaGetDevice");
    if (st != KVQ_OK) return st;
    if (dev < 0 || dev >= kMaxDevices)
        return kvq_set_error(KVQ_ERR_UNSUPPORTED, "kvq_decode_attn_int2_noalloc: device %d above %d", dev,
                             kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        st = kvq_check_cuda(cudaGetSymbolAddress(&p, g_decode_scratch),
                            "kvq_decode_attn_int2_noalloc: cudaGetSymbolAddress");
        if (st != KVQ_OK) return st;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KVQ_OK;
}

// Runs once the arguments have passed every check: the error word and the
// split tickets at the front of the scratch must start at zero.
kvq_status prepare_scratch(size_t zeroed, void* stream, void** ws) {
    void* scratch = nullptr;
    kvq_status st = scratch_address(&scratch);
    if (st != KVQ_OK) return st;
    st = kvq_check_cuda(cudaMemsetAsync(scratch, 0, zeroed, static_cast<cudaStream_t>(stream)),
                        "kvq_decode_attn_int2_noalloc: clearing scratch");
    if (st != KVQ_OK) return st;
    *ws = scratch;
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_int2_noalloc(const void* q, int B, int H_q, int H_kv, int d, const void* cache,
                                                   int64_t num_pages, const int32_t* block_table,
                                                   int max_pages_per_seq, const int32_t* context_lens,
                                                   const float* R_k, const float* R_v, float scale, float* out,
                                                   int num_splits, void* stream) {
    return kvq_decode_int2_checked("kvq_decode_attn_int2_noalloc", q, B, H_q, H_kv, d, cache, num_pages, block_table,
                                   max_pages_per_seq, context_lens, R_k, R_v, scale, out, num_splits, stream,
                                   kNoallocScratchBytes, prepare_scratch);
}
