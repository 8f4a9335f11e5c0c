// Tile helpers shared by the tensor-core chunked kernels: the byte layout of
// K-major fp16 operand tiles in the 128-byte swizzled canonical form that
// tcgen05 shared-memory descriptors describe, vector conversions into such
// tiles, and warp-level TF32 products for the small blocks of the
// triangular inverse.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn {
namespace ct {

// Byte offset of element (row, k) in a K-major, 128-byte swizzled fp16 tile with R rows.
__device__ __forceinline__ uint32_t sw(int row, int k, int R) {
    const int kb = k >> 6, kk = k & 63;
    return (uint32_t)(kb * R * 128 + row * 128 + ((((kk >> 3) ^ (row & 7)) & 7) << 4) + (kk & 7) * 2);
}

__device__ __forceinline__ void st_h(uint8_t *base, uint32_t off, float x) {
    *reinterpret_cast<__half *>(base + off) = __float2half_rn(x);
}

// Four consecutive elements (k % 4 == 0) of one row: one 8-byte store.
__device__ __forceinline__ void st_h4(uint8_t *base, uint32_t off, float a, float b, float c, float d) {
    __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&lo);
    v.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(base + off) = v;
}

template <typename T>
__device__ __forceinline__ void ld4(const T *p, float (&v)[4]);
template <>
__device__ __forceinline__ void ld4<float>(const float *p, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <>
__device__ __forceinline__ void ld4<__half>(const __half *p, float (&v)[4]) {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&x.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&x.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}


// 2^x on the special-function unit (relative error about 2^-22; flushes
// subnormal results to zero, which only negligible decay products reach).
// The chunked kernels keep cumulative log decays in log2 units so that each
// decay factor of A, P o D and the decayed deltas is one such instruction.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float LOG2E = 1.4426950408889634f;

// ---- Small products on the warp-level tensor cores
//
// The block products of the triangular inverse are 16 x 16 and 32 x 32: small
// and dependent, so a tcgen05 product per level is an asynchronous round trip
// (operand tiles, issue, mbarrier, tensor-memory read-back) -- measured, that
// variant made the prep kernel 200.9 us against 140.6 -- and on the CUDA
// cores they are bound by shared-memory traffic.  They run as mma.sync
// m16n8k8 TF32 products (10-bit mantissas, FP32 accumulation).  The inverse only feeds the tensor cores as an fp16 operand
// (also a 10-bit mantissa), and at the full varlen prefill (15,991 tokens)
// TF32 products gave the same end-to-end error against the FP64 oracle as
// FP32-accurate split products (output 8.10e-4, state 5.77e-4 vs 5.80e-4
// max-relative): the fp16 operand roundings dominate.

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One warp: the 16 x 8 tile C = X Y with X [16][K] (row stride xs) and
// Y [K][8] (row stride ys), both fp32 in shared memory; C written with the
// given sign to C_ (row stride cs).  m16n8k8 fragment layout: lane = 4 g + t;
// A holds (g, t), (g+8, t), (g, t+4), (g+8, t+4); B holds (t, g), (t+4, g);
// C holds (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1).
template <int K>
__device__ __forceinline__ void warp_tile_16x8(const float *X_, int xs, const float *Y_, int ys, float *C_, int cs,
                                               float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[4], bh[2];
        ah[0] = to_tf32(X_[g * xs + k0 + t]);
        ah[1] = to_tf32(X_[(g + 8) * xs + k0 + t]);
        ah[2] = to_tf32(X_[g * xs + k0 + t + 4]);
        ah[3] = to_tf32(X_[(g + 8) * xs + k0 + t + 4]);
        bh[0] = to_tf32(Y_[(k0 + t) * ys + g]);
        bh[1] = to_tf32(Y_[(k0 + t + 4) * ys + g]);
        mma_tf32(d, ah, bh);
    }
    C_[g * cs + 2 * t] = sign * d[0];
    C_[g * cs + 2 * t + 1] = sign * d[1];
    C_[(g + 8) * cs + 2 * t] = sign * d[2];
    C_[(g + 8) * cs + 2 * t + 1] = sign * d[3];
}


}  // namespace ct
}  // namespace gdn
