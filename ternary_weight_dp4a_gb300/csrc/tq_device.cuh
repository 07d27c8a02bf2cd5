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
// the 8-byte pool {b:a}, or, when sel bit 4i+3 is set, that byte's sign bit
// replicated over all eight bits.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while its predecessor in the stream still runs;
// pdl_wait() blocks until that predecessor has completed and its writes are
// visible (it returns at once when the launch had no such predecessor).
// Nothing the predecessor writes may be read, and nothing it reads may be
// written, before pdl_wait().
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA engine) helpers.  Every wait is bounded by a
// clock64 budget; a wait that runs out returns false and the caller records
// an error instead of spinning forever.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// try_wait without a suspend-time hint: the hardware may park the waiting
// thread for a short, system-defined time.  A long hint (tens of
// microseconds) parks waiters past the completion of phases that turn over
// every few hundred nanoseconds: the ring's slots at four or more rows per
// step, which then ran about 12% slower.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ~0.5 s at 2 GHz: far beyond any legitimate wait in these kernels
constexpr long long kWaitBudgetCycles = 1ll << 30;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitBudgetCycles) return false;
    return true;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Bulk copy global -> shared (16-byte aligned addresses, size a multiple of
// 16); completion is counted in bytes on the mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 policy for data read once: its lines are the first evicted, so a
// stream of them does not push out what other kernels reuse.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2D tensor copy global -> shared: the box at (x bytes, y rows) of the tensor
// described by *tmap (a kernel-parameter tensor map) lands densely at dst;
// completion is counted in bytes on `bar` (out-of-range parts read as zero);
// the lines are cached in L2 under `policy`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 3D tensor copy global -> shared: the box at (x, y, z) lands densely at dst
// (x fastest); completion counted in bytes on `bar`; L2 policy as above.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 16-bit read-only load (weight scales read outside the TMA path).
__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p) {
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Exact int -> float for |i| < 2^22 through the fp32 bit pattern of 2^23 + 2^22:
// (float)(i + bias) where `magic_minus_bias` = 0x4b400000 - bias.
__device__ __forceinline__ float int_to_float_exact(int i, int magic_minus_bias) {
    return __fsub_rn(__int_as_float(i + magic_minus_bias), 12582912.0f);
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
