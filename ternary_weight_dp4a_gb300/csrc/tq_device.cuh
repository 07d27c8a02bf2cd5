// tq_device.cuh -- device-side helpers shared by the libtq kernels (sm_103a).
//
// Every floating-point step uses explicit round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fmaf_rn, ...) so that no multiply-add is
// contracted and each rounding is the one the C ABI documents.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tq {

constexpr int kBlock = 128;        // weights per scale block / WHT size
constexpr int kLanesPerRow = 8;    // partial sums per output (fold order)
constexpr int kActStride = 144;    // staged activation bytes per block (128 + 16 pad)

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// prmt.b32 in its default mode: byte i of the result is byte sel[4i+2:4i] of
// the 8-byte pool {b:a}; sel bit 4i+3 must be 0 here (no sign replication).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// 32-byte streaming load of weight codes (read once: no L1 allocation).
struct u32x8 { uint32_t v[8]; };

__device__ __forceinline__ u32x8 ldg_stream_32B(const void *p) {
    u32x8 r;
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]),
                   "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_stream_16B(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p) {
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// exp and SiLU.  exp(z) = 2^n * P(r): Cody-Waite reduction with ln 2 split as
// L1 (ln 2 rounded to binary32 with its low 12 significand bits cleared) and
// L2 = ln 2 - L1, P = sum_{j<=7} r^j / j! by Horner's rule with fused
// multiply-adds (W. J. Cody, W. Waite, "Software Manual for the Elementary
// Functions", 1980).  Spelled out so the result is reproducible bit for bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float tq_expf(float z) {
    if (z != z) return z;
    if (z > 88.72283935546875f) return __int_as_float(0x7f800000);
    if (z < -103.972084045410156f) return 0.0f;
    const float kLog2e = __uint_as_float(0x3fb8aa3bu);
    const float kL1 = __uint_as_float(0x3f317000u);
    const float kL2 = __uint_as_float(0x3805fdf4u);
    const float n = rintf(__fmul_rn(z, kLog2e));
    float r = __fmaf_rn(-n, kL1, z);
    r = __fmaf_rn(-n, kL2, r);
    float p = __uint_as_float(0x39500d01u);                 // 1/7!
    p = __fmaf_rn(p, r, __uint_as_float(0x3ab60b61u));       // 1/6!
    p = __fmaf_rn(p, r, __uint_as_float(0x3c088889u));       // 1/5!
    p = __fmaf_rn(p, r, __uint_as_float(0x3d2aaaabu));       // 1/4!
    p = __fmaf_rn(p, r, __uint_as_float(0x3e2aaaabu));       // 1/3!
    p = __fmaf_rn(p, r, 0.5f);                               // 1/2!
    p = __fmaf_rn(p, r, 1.0f);                               // 1/1!
    p = __fmaf_rn(p, r, 1.0f);                               // 1/0!
    const int ni = static_cast<int>(n);
    const int n1 = ni / 2;          // truncates toward zero
    const int n2 = ni - n1;
    const float s1 = __int_as_float((n1 + 127) << 23);
    const float s2 = __int_as_float((n2 + 127) << 23);
    return __fmul_rn(__fmul_rn(p, s1), s2);
}

__device__ __forceinline__ float tq_silu(float g) {
    return __fdiv_rn(g, __fadd_rn(1.0f, tq_expf(-g)));
}

}  // namespace tq
