// INT2 group quantisation of rotated vectors, shared by every kernel that
// writes the INT2 cache (the append kernels and the fused decode step), so
// each writes the same bytes.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization" §1: all values of a
// group of 32 rotated channels share one scale; asymmetric levels min + code
// * scale with fp16 scale and min; clip ratio c of Q2(.; c, G) (§3.1 Eq. 4).
#pragma once

#include "kvq_common.cuh"

namespace kvq {

// Group parameters from the exact group min / max: the clip ratio c of
// Q2(.; c, G) scales both range ends, scale = (max - min) / 3 and min go
// to fp16 (saturating).
__device__ __forceinline__ void int2_params(float mn, float mx, float clip, __half& sh, __half& mh) {
    mn = __fmul_rn(clip, mn);
    mx = __fmul_rn(clip, mx);
    sh = f16_sat(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
    mh = f16_sat(mn);
}

// code = #{c : min + (c + 1/2) scale < x}, decided exactly
__device__ __forceinline__ int int2_code(float x, float mnf, float scf) {
    if (!(scf > 0.f)) return 0;
    float hi, lo;
    two_sum(x, -mnf, hi, lo);
    return (int)diff_gt(hi, lo, __fmul_rn(scf, 0.5f)) + (int)diff_gt(hi, lo, __fmul_rn(scf, 1.5f)) +
           (int)diff_gt(hi, lo, __fmul_rn(scf, 2.5f));
}

// The (scale, min) of slot s, group g: keys one word per group, values
// pair-major halves.
__device__ __forceinline__ void int2_store_meta(uint8_t* tile, int is_v, int s, int g, __half sh, __half mh) {
    if (is_v) {
        uint8_t* m = tile + vm_scale_off(s, g);
        *reinterpret_cast<__half*>(m) = sh;
        *reinterpret_cast<__half*>(m + VM_MINS) = mh;
    } else {
        const uint32_t meta = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(mh) << 16);
        *reinterpret_cast<uint32_t*>(tile + OFF_KM + 16 * s + 4 * g) = meta;
    }
}

// The code byte of a 32-channel group: lane l of the group's warp holds
// channel 32 g + l; byte 4 b + g of the record holds channels 32 g + 4 b + c
// at bits 2c (c = 0..3).  Returns the byte in lanes l % 4 == 0 (b = l / 4).
__device__ __forceinline__ uint32_t int2_gather_byte(int code, int lane) {
    uint32_t bits = (uint32_t)code << (2 * (lane & 3));
    bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
    bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
    return bits;
}

}  // namespace kvq
