// Block-GTQ append and decode kernels.
#include "kvq_common.cuh"

extern "C" kvq_status bgtq_append(const void*, const void*, int, int, int, const int32_t*, const int8_t*, int, int,
                                  const float*, const int64_t*, const double*, void*, int64_t, int32_t*, void*) {
    return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_append: not built yet");
}

extern "C" kvq_status bgtq_decode_attn(const void*, int, int, int, int, const void*, int64_t, const int32_t*, int,
                                       const int32_t*, const int8_t*, int, int, const float*, const int64_t*,
                                       const double*, float, float*, void*, size_t, int, void*) {
    return kvq_set_error(KVQ_ERR_UNSUPPORTED, "bgtq_decode_attn: not built yet");
}
