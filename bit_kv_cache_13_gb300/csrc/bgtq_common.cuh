// Block-GTQ pieces shared by the append, calibration and decode kernels:
// the per-head layout of the grouped key sub-vectors, the scaled codebook
// and the tile geometry.
//
// "RoPE-Aware Bit Allocation for KV-Cache Quantization", method step (3):
// RoPE blocks of equal width b form one sub-vector G_b, blocks ascending
// inside a group, each block as (dim i, dim i + d/2); the groups are laid
// out in ascending width in a dense LSB-first bit stream.
#pragma once

#include "merge.cuh"

namespace kvq {

// Per-head layout of the grouped key sub-vectors (built from the widths).
struct BgtqLayout {
    int16_t dim[D];      // gathered position -> original dimension
    int16_t start[9];    // first position of the width-b group
    int16_t n[9];        // length of the width-b group (2 * blocks)
    int16_t bitstart[9]; // first code bit of the width-b group
    int total_bits;      // sum over positions of the widths
    int ok;              // widths all in 1..8
};

// Thread 0 fills the layout: groups in ascending width, blocks ascending
// inside a group, each block as (dim i, dim i + 64).
__device__ __forceinline__ void build_layout(const int8_t* __restrict__ w, BgtqLayout& L) {
    int pos = 0, bit = 0, ok = 1;
    for (int i = 0; i < D / 2; ++i) ok &= (w[i] >= 1 && w[i] <= 8);
    for (int b = 1; b <= 8; ++b) {
        L.start[b] = (int16_t)pos;
        L.bitstart[b] = (int16_t)bit;
        for (int i = 0; i < D / 2; ++i)
            if (w[i] == b) {
                L.dim[pos++] = (int16_t)i;
                L.dim[pos++] = (int16_t)(i + D / 2);
            }
        L.n[b] = (int16_t)(pos - L.start[b]);
        bit += b * L.n[b];
    }
    L.total_bits = bit;
    L.ok = ok && pos == D;
}

__host__ __device__ inline int bgtq_kb(int total_bits) { return 4 * ((2 * total_bits + 31) / 32); }

// Scaled codebook fp32(C_b[c] / sqrt(n)), computed in fp64 then rounded once.
__device__ __forceinline__ float scaled_centroid(const double* __restrict__ cb, int b, int c, int n) {
    return __double2float_rn(cb[(b - 1) * 256 + c] / sqrt((double)n));
}

// Number of midpoints (c_k + c_{k+1}) / 2 (exact in fp64) strictly below y:
// the nearest centroid, ties to the lower index.
__device__ __forceinline__ int nearest_code(float y, const float* __restrict__ c, int levels) {
    int lo = 0, hi = levels - 1;
    const double yd = (double)y;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const double m = 0.5 * ((double)c[mid] + (double)c[mid + 1]);
        if (m < yd) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Group of gathered position p (1..8).
__device__ __forceinline__ int group_of(const BgtqLayout& L, int p) {
    int b = 1;
    while (b < 8 && !(p >= L.start[b] && p < L.start[b] + L.n[b])) ++b;
    return b;
}


// Tile of one (page, KV head): K codes 16 x KB, K norms 16 x 16 (one fp16 per
// width 1..8), V codes 16 x VB (VB = 16 v_bits), V norms 16 x 2.
struct BgtqTile {
    int kb, vb, off_kn, off_vc, off_vn, bytes;
    __host__ __device__ BgtqTile(int total_bits, int v_bits)
        : kb(bgtq_kb(total_bits)), vb(16 * v_bits), off_kn(PAGE * bgtq_kb(total_bits)),
          off_vc(PAGE * bgtq_kb(total_bits) + PAGE * 16), off_vn(PAGE * bgtq_kb(total_bits) + PAGE * 16 + PAGE * 16 * v_bits),
          bytes(PAGE * (bgtq_kb(total_bits) + 16 + 16 * v_bits + 2)) {}
};

}  // namespace kvq

// Argument checks shared by the Block-GTQ entry points.
kvq_status bgtq_check_common(const char* fn, int d, int H_kv, int total_bits, int v_bits, const float* pi_table);
