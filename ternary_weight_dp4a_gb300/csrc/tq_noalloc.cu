// tq_noalloc.cu -- tq_ffn_step_static: the FFN decode step for callers that
// cannot hand the library a workspace.  Its scratch lives in a fixed array
// compiled into the library; the call itself allocates nothing.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_workspace.h"

namespace {

// Largest sizes the built-in scratch serves.
constexpr int kStaticMaxRows = TQ_STATIC_MAX_ROWS;
constexpr int kStaticMaxHidden = TQ_STATIC_MAX_HIDDEN;
constexpr int kStaticMaxInter = TQ_STATIC_MAX_INTER;

// The dp4a kernel's part of the FFN workspace at the largest sizes (the step
// this entry point runs; laid out as tq_ffn_step lays it out).
constexpr size_t kStaticBytes = tq::ffn_layout(kStaticMaxRows, kStaticMaxHidden, kStaticMaxInter).dp4a_total;

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
tq_status ffn_step_dp4a(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                        int32_t m, float *y, void *workspace, cudaStream_t str);
tq_status ffn_check_args(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                         int32_t m, const float *y);
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
    tq_status st = tq::ffn_check_args(gate, up, down, x, m, y);
    if (st != TQ_OK) return st;
    const int hidden = gate->k, inter = gate->n;
    if (m > kStaticMaxRows || hidden > kStaticMaxHidden || inter > kStaticMaxInter)
        return TQ_ERR_UNSUPPORTED;               // beyond the built-in scratch
    const size_t need = tq::ffn_layout(m, hidden, inter).dp4a_total;
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
    return tq::ffn_step_dp4a(gate, up, down, x, m, y, ws, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
