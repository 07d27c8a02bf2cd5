// tq_noalloc.cu -- tq_ffn_step_static: the FFN decode step for callers that
// cannot hand the library a workspace.  Its scratch lives in a fixed array
// compiled into the library; the call itself allocates nothing.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "tq.h"

namespace {

// Largest sizes the built-in scratch serves.
constexpr int kStaticMaxRows = TQ_STATIC_MAX_ROWS;
constexpr int kStaticMaxHidden = TQ_STATIC_MAX_HIDDEN;
constexpr int kStaticMaxInter = TQ_STATIC_MAX_INTER;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The FFN workspace at the largest sizes, laid out as tq_ffn_step lays it out
// (every section 256-byte aligned): qx, sx, h, qh, sh, counters, ybuf, err,
// sync counters, staged h and its (scale, magic - sum) pairs, h after the
// first butterfly stages.
constexpr size_t kStaticBytes =
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxHidden) +
    align256(static_cast<size_t>(kStaticMaxRows) * (kStaticMaxHidden / 128) * 4) +
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxInter * 2) +
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxInter) +
    align256(static_cast<size_t>(kStaticMaxRows) * (kStaticMaxInter / 128) * 4) +
    align256(static_cast<size_t>(kStaticMaxInter / 128) * 4) +
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxHidden * 4) + align256(4) +
    align256(static_cast<size_t>(2 + kStaticMaxInter / 1024) * 4) +
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxInter) +
    align256(static_cast<size_t>(kStaticMaxRows) * (kStaticMaxInter / 128) * 8) +
    align256(static_cast<size_t>(kStaticMaxRows) * kStaticMaxInter * 4);

// One copy per GPU that loads the library, held until the process exits.
// Device code could name it directly; host code must use the address from
// cudaGetSymbolAddress (its name on the host is only a stand-in).
static __device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_addr[kMaxDevices] = {};

}  // namespace

namespace tq {
void record_cuda_error(int e);
}

namespace {
tq_status fail_cuda(cudaError_t e) {
    tq::record_cuda_error(static_cast<int>(e));
    return TQ_ERR_CUDA;
}
}  // namespace

extern "C" {

size_t tq_ffn_static_workspace_bytes(void) { return kStaticBytes; }

tq_status tq_ffn_step_static(const tq_weight *gate, const tq_weight *up, const tq_weight *down,
                             const uint16_t *x, int32_t m, float *y, tq_stream_t stream) {
    if (gate == nullptr || up == nullptr || down == nullptr || x == nullptr || y == nullptr)
        return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    const int hidden = gate->k, inter = gate->n;
    if (m > kStaticMaxRows || hidden > kStaticMaxHidden || inter > kStaticMaxInter)
        return TQ_ERR_UNSUPPORTED;               // beyond the built-in scratch
    const size_t need = tq_ffn_workspace_bytes(m, hidden, inter);
    if (need == 0) return TQ_ERR_INVALID_ARG;
    if (need > kStaticBytes) return TQ_ERR_UNSUPPORTED;

    // set-up, once per device, with that device current: the array's device
    // address
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_addr[dev] == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_static_workspace);
            if (e != cudaSuccess) return fail_cuda(e);
            g_addr[dev] = p;
        }
        ws = g_addr[dev];
    }
    // The array keeps the last call's contents: zero it (an async memset on
    // the caller's stream, no allocation) so the completion counters and the
    // error and barrier words start at zero.
    e = cudaMemsetAsync(ws, 0, need, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    return tq_ffn_step(gate, up, down, x, m, y, ws, need, stream);
}

}  // extern "C"
