// tq_mma_rate.cu -- throughput of tcgen05.mma kind::f8f6f4 (e4m3 x e4m3,
// f32 accumulators in tensor memory) at M = 128, K = 32 per instruction, for
// N = 16, 64, 128, 256 and the A operand in tensor memory or in shared
// memory.  Every SM runs one CTA; one thread issues 8 x 4 MMAs per
// iteration into 8 accumulators and waits for their commit, 200 iterations.
// The figure that decides a ternary GEMV on the tensor cores is the time per
// MMA at small N: it fixes how many weight bytes (the A operand, one e4m3
// byte per weight) the tensor core can take per cycle.
//
// Every tensor-memory column is written before use, accumulators are
// 32-column aligned, and every wait is bounded (error flags instead of a
// hang).  Build: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o
// tq_mma_rate tq_mma_rate.cu
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include <cuda_runtime.h>

#define CK(x)                                                                                \
    do {                                                                                     \
        cudaError_t e_ = (x);                                                                \
        if (e_ != cudaSuccess) {                                                             \
            printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_));             \
            exit(1);                                                                         \
        }                                                                                    \
    } while (0)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > (1ll << 31)) return false;
    return true;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: no swizzle, K-major core matrices of 8 rows x 16 bytes
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3ffff) >> 4);
    d |= static_cast<uint64_t>(lbo >> 4) << 16;
    d |= static_cast<uint64_t>(sbo >> 4) << 32;
    d |= 1ull << 46;
    return d;
}
// instruction descriptor: f32 accumulator, e4m3 A and B, N >> 3, M >> 4
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// mode bit 0: A from shared memory (else tensor memory).
__global__ void __launch_bounds__(128, 1) rate(int iters, int N, int mode, unsigned *err, long long *cycles) {
    extern __shared__ __align__(1024) uint8_t sm[];
    uint8_t *sA = sm;              // 128 rows x 128 bytes
    uint8_t *sB = sm + 16384;      // N rows x 128 bytes
    __shared__ __align__(8) uint64_t bar, done;
    __shared__ uint32_t tmem;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_init(smem_u32(&done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = threadIdx.x; i < (16384 + N * 128) / 4; i += 128) reinterpret_cast<uint32_t *>(sm)[i] = 0x38383838u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem;
    // every column: A region [0, 256) holds e4m3 1.0, D region [256, 512) zero
    {
        const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
        for (int c0 = 0; c0 < 512; c0 += 32) {
            const uint32_t v = c0 < 256 ? 0x38383838u : 0u;
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
                "%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(tb + lb + c0),
                "r"(v)
                : "memory");
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int dstride = N < 32 ? 32 : N;
    const int nd = 256 / dstride;
    const uint32_t idesc = idesc_e4m3(128, N);
    long long t0 = 0, t1 = 0;
    if (threadIdx.x == 0) {
        int commits = 0;
        t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            for (int blk = 0; blk < 8; ++blk) {
                const uint32_t d = tb + 256 + (blk % nd) * dstride;
                for (int i = 0; i < 4; ++i) {
                    const uint64_t bd = sdesc(smem_u32(sB) + i * 2 * (N / 8) * 128, (N / 8) * 128, 128);
                    if (mode & 1) {
                        const uint64_t ad = sdesc(smem_u32(sA) + i * 2 * 128, 128, 1024);
                        asm volatile(
                            "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
                            "l"(ad), "l"(bd), "r"(idesc), "r"(i > 0 ? 1 : 0)
                            : "memory");
                    } else {
                        const uint32_t at = tb + (blk % 8) * 32 + 8 * i;
                        asm volatile(
                            "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p; }" ::"r"(d),
                            "r"(at), "l"(bd), "r"(idesc), "r"(i > 0 ? 1 : 0)
                            : "memory");
                    }
                }
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar))
                         : "memory");
            if (!mbar_wait(smem_u32(&bar), commits & 1)) atomicOr(err, 1u);
            ++commits;
        }
        t1 = clock64();
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&done))
                     : "memory");
    }
    __syncwarp();
    if (!mbar_wait(smem_u32(&done), 0)) atomicOr(err, 2u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb) : "memory");
}

int main() {
    unsigned *derr;
    long long *dcyc;
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    CK(cudaMalloc(&derr, 4));
    CK(cudaMalloc(&dcyc, sizeof(long long) * sms));
    CK(cudaFuncSetAttribute(rate, cudaFuncAttributeMaxDynamicSharedMemorySize, 131072));
    long long *cyc = static_cast<long long *>(malloc(sizeof(long long) * sms));
    const int iters = 200;
    for (int mode = 0; mode < 2; ++mode)
        for (int N : {16, 64, 128, 256}) {
            CK(cudaMemset(derr, 0, 4));
            rate<<<sms, 128, 131072>>>(iters, N, mode, derr, dcyc);
            CK(cudaGetLastError());
            CK(cudaDeviceSynchronize());
            unsigned herr;
            CK(cudaMemcpy(cyc, dcyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost));
            CK(cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost));
            double mean = 0;
            for (int i = 0; i < sms; ++i) mean += static_cast<double>(cyc[i]);
            mean /= sms;
            const double per = mean / (iters * 8.0 * 4.0);
            printf("A in %s N=%3d: err=%u  %.1f cycles per MMA (M128 K32, %d SMs)  %.1f B/cycle of A  %.0f MACs/cycle/SM\n",
                   mode ? "SMEM" : "TMEM", N, herr, per, sms, 4096.0 / per, 128.0 * N * 32 / per);
        }
    free(cyc);
    return 0;
}
