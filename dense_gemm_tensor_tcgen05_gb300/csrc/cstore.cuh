// cstore.cuh -- reading and writing elements of C in its storage type.
//
// C holds FP32, FP16 or BF16 (gemm_options_t.c_dtype).  Every kernel forms
// its results in FP32 (the product, then alpha * AB + beta * C) and, for a
// 16-bit C, rounds each result once to nearest, ties to even, as it stores
// it.  A 16-bit C read for beta * C is widened to FP32 exactly.
#pragma once

#include <cstdint>

namespace gb300 {

constexpr int kCF32 = 0, kCF16 = 1, kCBF16 = 2;

// Two FP32 values rounded to the 16-bit type and packed; `lo` lands in the
// low half (the lower address).  cvt.rn.{f16,bf16}x2.f32 puts its first
// source in the upper half.
__device__ __forceinline__ uint32_t c_pack2(float lo, float hi, int ct) {
    uint32_t r;
    if (ct == kCF16)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float c_widen(uint16_t h, int ct) {
    if (ct == kCF16) {
        float f;
        asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
        return f;
    }
    return __uint_as_float(static_cast<uint32_t>(h) << 16);   // BF16 is FP32's upper half
}

// Element i of C (i = row * ldc + column).
__device__ __forceinline__ float c_load(const void* C, int64_t i, int ct) {
    if (ct == kCF32) return static_cast<const float*>(C)[i];
    return c_widen(static_cast<const uint16_t*>(C)[i], ct);
}

__device__ __forceinline__ void c_store(void* C, int64_t i, float v, int ct) {
    if (ct == kCF32)
        static_cast<float*>(C)[i] = v;
    else
        static_cast<uint16_t*>(C)[i] = static_cast<uint16_t>(c_pack2(v, 0.0f, ct) & 0xFFFFu);
}

// Four consecutive elements from i: one 16-byte access for FP32, one 8-byte
// access for 16-bit types.  The caller guarantees that alignment (C's base
// and ldc, with i a multiple of 4).
__device__ __forceinline__ float4 c_load4(const void* C, int64_t i, int ct) {
    if (ct == kCF32) return *reinterpret_cast<const float4*>(static_cast<const float*>(C) + i);
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(C) + i);
    return make_float4(c_widen(static_cast<uint16_t>(w.x & 0xFFFFu), ct),
                       c_widen(static_cast<uint16_t>(w.x >> 16), ct),
                       c_widen(static_cast<uint16_t>(w.y & 0xFFFFu), ct),
                       c_widen(static_cast<uint16_t>(w.y >> 16), ct));
}

__device__ __forceinline__ void c_store4(void* C, int64_t i, float a, float b, float c, float d,
                                         int ct) {
    if (ct == kCF32) {
        *reinterpret_cast<float4*>(static_cast<float*>(C) + i) = make_float4(a, b, c, d);
    } else {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(C) + i) =
            make_uint2(c_pack2(a, b, ct), c_pack2(c, d, ct));
    }
}

// Bytes of one element of C.
__host__ __device__ constexpr int c_elem_bytes(int ct) { return ct == kCF32 ? 4 : 2; }

}  // namespace gb300
