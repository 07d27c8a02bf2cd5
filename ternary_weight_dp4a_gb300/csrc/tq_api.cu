// tq_api.cu -- the C ABI of libtq (declared in include/tq.h): argument checks,
// workspace layout and kernel dispatch.  Every data pointer is a device
// pointer owned by the caller; nothing here allocates.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_launch.h"
#include "tq_misc.cuh"
#include "tq_rotq.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

tq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    g_last_cuda_error = static_cast<int>(e);
    return TQ_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kWsAlign = 256;

struct FfnWorkspace {
    size_t qx, sx, h, qh, sh, total;
};

FfnWorkspace ffn_layout(int64_t m, int64_t hidden, int64_t inter) {
    FfnWorkspace w{};
    size_t off = 0;
    w.qx = off; off = round_up(off + static_cast<size_t>(m * hidden), kWsAlign);
    w.sx = off; off = round_up(off + static_cast<size_t>(m * (hidden / 128)) * 4, kWsAlign);
    w.h = off;  off = round_up(off + static_cast<size_t>(m * inter) * 2, kWsAlign);
    w.qh = off; off = round_up(off + static_cast<size_t>(m * inter), kWsAlign);
    w.sh = off; off = round_up(off + static_cast<size_t>(m * (inter / 128)) * 4, kWsAlign);
    w.total = off;
    return w;
}

tq_status check_weight(const tq_weight *w) {
    if (w == nullptr || w->codes == nullptr || w->scales == nullptr) return TQ_ERR_INVALID_ARG;
    if (w->n < 1 || w->k < 128 || w->k % 128 != 0) return TQ_ERR_INVALID_ARG;
    if (w->fmt != TQ_FMT_TERNARY2 && w->fmt != TQ_FMT_BINARY1) return TQ_ERR_INVALID_ARG;
    if (!aligned(w->codes, 32) || !aligned(w->scales, 2)) return TQ_ERR_ALIGNMENT;
    return TQ_OK;
}

tq_status check_smem(int fmt, int m, int k) {
    const size_t need = tq::gemv_smem_bytes(fmt, m, k / 128);
    cudaError_t e = cudaSuccess;
    const size_t have = tq::max_smem_optin(&e);
    if (e != cudaSuccess) return cuda_status(e);
    return need <= have ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

cudaError_t launch_gemv(const tq::GemvArgs &a, int fmt, int m, int nw, cudaStream_t stream) {
    return fmt == TQ_FMT_TERNARY2 ? tq::launch_gemv_t2(a, m, nw, stream)
                                  : tq::launch_gemv_b1(a, m, nw, stream);
}

cudaError_t launch_gateup(const tq_weight *gate, const tq_weight *up, const int8_t *qx,
                          const float *sx, int m, uint16_t *h, cudaStream_t stream) {
    tq::GemvArgs gu{};
    gu.codes[0] = gate->codes;
    gu.codes[1] = up->codes;
    gu.scales[0] = gate->scales;
    gu.scales[1] = up->scales;
    gu.n = gate->n;
    gu.k = gate->k;
    gu.q = qx;
    gu.s = sx;
    gu.h = h;
    return launch_gemv(gu, gate->fmt, m, 2, stream);
}

cudaError_t launch_rotq(const uint16_t *x, int64_t m, int k, int8_t *q, float *s,
                        cudaStream_t stream) {
    const int64_t blocks = m * (k / 128);
    const int64_t warps_per_cta = 256 / 32;
    const unsigned grid = static_cast<unsigned>((blocks + warps_per_cta - 1) / warps_per_cta);
    tq::rotate_quant_kernel<<<grid, 256, 0, stream>>>(x, blocks, k, q, s);
    return cudaGetLastError();
}

}  // namespace

namespace tq {
size_t max_smem_optin(cudaError_t *err) {
    int dev = 0, v = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != nullptr) *err = e;
    return e == cudaSuccess ? static_cast<size_t>(v) : 0;
}
}  // namespace tq

extern "C" {

const char *tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_ALIGNMENT: return "misaligned pointer";
        case TQ_ERR_UNSUPPORTED: return "unsupported size";
        case TQ_ERR_WORKSPACE: return "workspace too small";
        case TQ_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int tq_last_cuda_error(void) { return g_last_cuda_error; }

tq_status tq_pack_weights(const uint8_t *codes, int32_t n, int32_t k, int32_t fmt,
                          uint8_t *packed, tq_stream_t stream) {
    if (codes == nullptr || packed == nullptr) return TQ_ERR_INVALID_ARG;
    if (n < 1 || k < 128 || k % 128 != 0) return TQ_ERR_INVALID_ARG;
    if (fmt != TQ_FMT_TERNARY2 && fmt != TQ_FMT_BINARY1) return TQ_ERR_INVALID_ARG;
    if (!aligned(packed, 32)) return TQ_ERR_ALIGNMENT;
    const int64_t out_bytes = static_cast<int64_t>(n) * k / (fmt == TQ_FMT_TERNARY2 ? 4 : 8);
    const int64_t want = (out_bytes + 255) / 256;
    const unsigned grid = static_cast<unsigned>(want < 65536 ? want : 65536);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (fmt == TQ_FMT_TERNARY2)
        tq::pack_kernel<0><<<grid, 256, 0, st>>>(codes, out_bytes, packed);
    else
        tq::pack_kernel<1><<<grid, 256, 0, st>>>(codes, out_bytes, packed);
    return cuda_status(cudaGetLastError());
}

tq_status tq_rotate_quant(const uint16_t *x, int32_t m, int32_t k, int8_t *q, float *s,
                          tq_stream_t stream) {
    if (x == nullptr || q == nullptr || s == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || k < 128 || k % 128 != 0) return TQ_ERR_INVALID_ARG;
    return cuda_status(launch_rotq(x, m, k, q, s, reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_gemv(const tq_weight *w, const int8_t *q, const float *s, int32_t m, float *y,
                  int32_t *blockdots, tq_stream_t stream) {
    tq_status st = check_weight(w);
    if (st != TQ_OK) return st;
    if (q == nullptr || s == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(s, 4) || !aligned(y, 4) || !aligned(blockdots, 4))
        return TQ_ERR_ALIGNMENT;
    st = check_smem(w->fmt, m, w->k);
    if (st != TQ_OK) return st;
    tq::GemvArgs a{};
    a.codes[0] = a.codes[1] = w->codes;
    a.scales[0] = a.scales[1] = w->scales;
    a.n = w->n;
    a.k = w->k;
    a.q = q;
    a.s = s;
    a.y = y;
    a.dots = blockdots;
    return cuda_status(launch_gemv(a, w->fmt, m, 1, reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_ffn_gateup(const tq_weight *gate, const tq_weight *up, const int8_t *qx,
                        const float *sx, int32_t m, uint16_t *h, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(gate)) != TQ_OK) return st;
    if ((st = check_weight(up)) != TQ_OK) return st;
    if (qx == nullptr || sx == nullptr || h == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (up->n != gate->n || up->k != gate->k || up->fmt != gate->fmt) return TQ_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(sx, 4) || !aligned(h, 2)) return TQ_ERR_ALIGNMENT;
    if ((st = check_smem(gate->fmt, m, gate->k)) != TQ_OK) return st;
    return cuda_status(launch_gateup(gate, up, qx, sx, m, h, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_ffn_workspace_bytes(int32_t m, int32_t hidden, int32_t inter) {
    if (m < 1 || hidden < 1 || inter < 1) return 0;
    return ffn_layout(m, hidden, inter).total;
}

tq_status tq_ffn_step(const tq_weight *gate, const tq_weight *up, const tq_weight *down,
                      const uint16_t *x, int32_t m, float *y, void *workspace,
                      size_t workspace_bytes, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(gate)) != TQ_OK) return st;
    if ((st = check_weight(up)) != TQ_OK) return st;
    if ((st = check_weight(down)) != TQ_OK) return st;
    if (x == nullptr || y == nullptr || workspace == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    const int hidden = gate->k, inter = gate->n;
    if (up->n != inter || up->k != hidden || down->n != hidden || down->k != inter)
        return TQ_ERR_INVALID_ARG;
    if (up->fmt != gate->fmt || down->fmt != gate->fmt) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4) || !aligned(workspace, kWsAlign)) return TQ_ERR_ALIGNMENT;
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if (workspace_bytes < L.total) return TQ_ERR_WORKSPACE;
    if ((st = check_smem(gate->fmt, m, hidden)) != TQ_OK) return st;
    if ((st = check_smem(gate->fmt, m, inter)) != TQ_OK) return st;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int8_t *qx = reinterpret_cast<int8_t *>(ws + L.qx);
    float *sx = reinterpret_cast<float *>(ws + L.sx);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    int8_t *qh = reinterpret_cast<int8_t *>(ws + L.qh);
    float *sh = reinterpret_cast<float *>(ws + L.sh);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    cudaError_t e = launch_rotq(x, m, hidden, qx, sx, s);
    if (e != cudaSuccess) return cuda_status(e);

    e = launch_gateup(gate, up, qx, sx, m, h, s);
    if (e != cudaSuccess) return cuda_status(e);

    e = launch_rotq(h, m, inter, qh, sh, s);
    if (e != cudaSuccess) return cuda_status(e);

    tq::GemvArgs dn{};
    dn.codes[0] = dn.codes[1] = down->codes;
    dn.scales[0] = dn.scales[1] = down->scales;
    dn.n = hidden;
    dn.k = inter;
    dn.q = qh;
    dn.s = sh;
    dn.y = y;
    return cuda_status(launch_gemv(dn, gate->fmt, m, 1, s));
}

tq_status tq_rmsnorm_bf16(const float *y, int32_t m, int32_t n, float eps, uint16_t *x_out,
                          tq_stream_t stream) {
    if (y == nullptr || x_out == nullptr || m < 1 || n < 1) return TQ_ERR_INVALID_ARG;
    tq::rmsnorm_bf16_kernel<<<m, tq::kNormThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        y, n, eps, x_out);
    return cuda_status(cudaGetLastError());
}

}  // extern "C"
