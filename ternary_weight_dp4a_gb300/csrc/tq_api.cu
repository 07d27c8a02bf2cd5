// tq_api.cu -- the C ABI of libtq (declared in include/tq.h): argument checks,
// workspace layout and kernel dispatch.  Every data pointer is a device
// pointer owned by the caller; nothing here allocates.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_fused_launch.h"
#include "tq_launch.h"
#include "tq_misc.cuh"
#include "tq_norm_kernels.cuh"

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

// Workspace of the FFN step / stack, each section 256-byte aligned:
//   qx int8 [m][hidden] | sx f32 [m][hidden/128] | h bf16 [m][inter] |
//   qh int8 [m][inter]  | sh f32 [m][inter/128]  | counters u32 [inter/128] |
//   ybuf f32 [m][hidden] | err u32 (nonzero: a kernel's bounded wait ran out) |
//   gbar u32[2] (grid barrier of the fused kernel)
struct FfnWorkspace {
    size_t qx, sx, h, qh, sh, counters, ybuf, err, gbar, total;
};

FfnWorkspace ffn_layout(int64_t m, int64_t hidden, int64_t inter) {
    FfnWorkspace w{};
    size_t off = 0;
    w.qx = off; off = round_up(off + static_cast<size_t>(m * hidden), kWsAlign);
    w.sx = off; off = round_up(off + static_cast<size_t>(m * (hidden / 128)) * 4, kWsAlign);
    w.h = off;  off = round_up(off + static_cast<size_t>(m * inter) * 2, kWsAlign);
    w.qh = off; off = round_up(off + static_cast<size_t>(m * inter), kWsAlign);
    w.sh = off; off = round_up(off + static_cast<size_t>(m * (inter / 128)) * 4, kWsAlign);
    w.counters = off; off = round_up(off + static_cast<size_t>(inter / 128) * 4, kWsAlign);
    w.ybuf = off; off = round_up(off + static_cast<size_t>(m * hidden) * 4, kWsAlign);
    w.err = off; off = round_up(off + 4, kWsAlign);
    w.gbar = off; off = round_up(off + 8, kWsAlign);
    w.total = off;
    return w;
}

struct FfnPtrs {
    int8_t *qx;
    float *sx;
    uint16_t *h;
    int8_t *qh;
    float *sh;
    unsigned *counters;
    float *ybuf;
    unsigned *err;
    unsigned *gbar;
};

FfnPtrs ffn_ptrs(void *ws, const FfnWorkspace &L) {
    uint8_t *b = static_cast<uint8_t *>(ws);
    return FfnPtrs{reinterpret_cast<int8_t *>(b + L.qx), reinterpret_cast<float *>(b + L.sx),
                   reinterpret_cast<uint16_t *>(b + L.h), reinterpret_cast<int8_t *>(b + L.qh),
                   reinterpret_cast<float *>(b + L.sh), reinterpret_cast<unsigned *>(b + L.counters),
                   reinterpret_cast<float *>(b + L.ybuf), reinterpret_cast<unsigned *>(b + L.err),
                   reinterpret_cast<unsigned *>(b + L.gbar)};
}

tq_status check_weight(const tq_weight *w) {
    if (w == nullptr || w->codes == nullptr || w->scales == nullptr) return TQ_ERR_INVALID_ARG;
    if (w->n < 1 || w->k < 128 || w->k % 128 != 0) return TQ_ERR_INVALID_ARG;
    if (w->fmt != TQ_FMT_TERNARY2 && w->fmt != TQ_FMT_BINARY1) return TQ_ERR_INVALID_ARG;
    if (!aligned(w->codes, 32) || !aligned(w->scales, 2)) return TQ_ERR_ALIGNMENT;
    return TQ_OK;
}

tq_status check_smem(int fmt, int m, bool gateup, int k, int n) {
    const size_t need = tq::gemv_smem_needed(fmt, m, gateup, k, n);
    cudaError_t e = cudaSuccess;
    const size_t have = tq::max_smem_optin(&e);
    if (e != cudaSuccess) return cuda_status(e);
    // the kernels' static shared memory (mbarriers, flags) is well under 1 KB
    return need + 1024 <= have ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

// gate [inter][hidden], up [inter][hidden], down [hidden][inter], one format
tq_status check_ffn(const tq_weight *gate, const tq_weight *up, const tq_weight *down, int m) {
    tq_status st;
    if ((st = check_weight(gate)) != TQ_OK) return st;
    if ((st = check_weight(up)) != TQ_OK) return st;
    if ((st = check_weight(down)) != TQ_OK) return st;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    const int hidden = gate->k, inter = gate->n;
    if (up->n != inter || up->k != hidden || down->n != hidden || down->k != inter)
        return TQ_ERR_INVALID_ARG;
    if (up->fmt != gate->fmt || down->fmt != gate->fmt) return TQ_ERR_INVALID_ARG;
    return TQ_OK;
}

// device limits last: every host-side check comes first
tq_status check_ffn_smem(int fmt, int m, int hidden, int inter) {
    tq_status st = check_smem(fmt, m, true, hidden, inter);
    return st != TQ_OK ? st : check_smem(fmt, m, false, inter, hidden);
}

tq_status check_ws(void *ws, size_t bytes, int m, int hidden, int inter) {
    if (ws == nullptr) return TQ_ERR_INVALID_ARG;
    if (!aligned(ws, kWsAlign)) return TQ_ERR_ALIGNMENT;
    if (bytes < ffn_layout(m, hidden, inter).total) return TQ_ERR_WORKSPACE;
    return TQ_OK;
}

cudaError_t launch_gemv(const tq::GemvArgs &a, int fmt, int m, bool gateup, cudaStream_t stream) {
    return fmt == TQ_FMT_TERNARY2 ? tq::launch_gemv_t2(a, m, gateup, stream)
                                  : tq::launch_gemv_b1(a, m, gateup, stream);
}

cudaError_t launch_rotq(const uint16_t *x, int64_t m, int k, int8_t *q, float *s,
                        cudaStream_t stream) {
    const int64_t blocks = m * (k / 128);
    const int64_t warps_per_cta = 256 / 32;
    const unsigned grid = static_cast<unsigned>((blocks + warps_per_cta - 1) / warps_per_cta);
    return tq::launch_pdl(tq::rotate_quant_kernel, dim3(grid), dim3(256), 0, stream, x, blocks, k,
                          q, s);
}

cudaError_t launch_gateup(const tq_weight *gate, const tq_weight *up, const int8_t *qx,
                          const float *sx, int m, uint16_t *h, int8_t *qh, float *sh,
                          unsigned *counters, unsigned *err, cudaStream_t stream) {
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
    gu.qh = qh;
    gu.sh = sh;
    gu.counters = counters;
    gu.err = err;
    return launch_gemv(gu, gate->fmt, m, true, stream);
}

cudaError_t launch_down(const tq_weight *down, const int8_t *qh, const float *sh, int m, float *y,
                        unsigned *err, cudaStream_t stream) {
    tq::GemvArgs dn{};
    dn.codes[0] = dn.codes[1] = down->codes;
    dn.scales[0] = dn.scales[1] = down->scales;
    dn.n = down->n;
    dn.k = down->k;
    dn.q = qh;
    dn.s = sh;
    dn.y = y;
    dn.err = err;
    return launch_gemv(dn, down->fmt, m, false, stream);
}

bool use_fused(int fmt, int m, int hidden, int inter) {
    if (!tq::fused_supported(fmt, m, hidden, inter)) return false;
    cudaError_t e = cudaSuccess;
    const size_t have = tq::max_smem_optin(&e);
    return e == cudaSuccess && tq::fused_smem(fmt, m, hidden, inter) + 1024 <= have;
}

tq::FfnFusedArgs fused_args(const FfnPtrs &P, int hidden, int inter, float eps) {
    tq::FfnFusedArgs f{};
    f.hidden = hidden;
    f.inter = inter;
    f.eps = eps;
    f.ybuf = P.ybuf;
    f.qx = P.qx;
    f.sx = P.sx;
    f.h = P.h;
    f.qh = P.qh;
    f.sh = P.sh;
    f.counters = P.counters;
    f.gbar = P.gbar;
    f.err = P.err;
    return f;
}

void set_layer(tq::FfnFusedArgs &f, int i, const tq_weight *g, const tq_weight *u, const tq_weight *d) {
    const tq_weight *w[3] = {g, u, d};
    for (int j = 0; j < 3; ++j) {
        f.layer[i].codes[j] = w[j]->codes;
        f.layer[i].scales[j] = w[j]->scales;
    }
}

}  // namespace

namespace tq {
// lets other translation units report through tq_last_cuda_error()
void record_cuda_error(int e) { g_last_cuda_error = e; }

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
    st = check_smem(w->fmt, m, false, w->k, w->n);
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
    return cuda_status(launch_gemv(a, w->fmt, m, false, reinterpret_cast<cudaStream_t>(stream)));
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
    if ((st = check_smem(gate->fmt, m, true, gate->k, gate->n)) != TQ_OK) return st;
    return cuda_status(launch_gateup(gate, up, qx, sx, m, h, nullptr, nullptr, nullptr, nullptr,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_ffn_workspace_bytes(int32_t m, int32_t hidden, int32_t inter) {
    if (m < 1 || hidden < 1 || inter < 1) return 0;
    return ffn_layout(m, hidden, inter).total;
}

tq_status tq_ffn_workspace_init(void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (workspace == nullptr) return TQ_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_ffn_stage_input(const uint16_t *x, int32_t m, int32_t hidden, int32_t inter,
                             void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (x == nullptr || m < 1 || m > TQ_MAX_ROWS || hidden < 128 || hidden % 128 != 0 ||
        inter < 128 || inter % 128 != 0)
        return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16)) return TQ_ERR_ALIGNMENT;
    tq_status st = check_ws(workspace, workspace_bytes, m, hidden, inter);
    if (st != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    return cuda_status(launch_rotq(x, m, hidden, P.qx, P.sx, reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_ffn_stage_gateup(const tq_weight *gate, const tq_weight *up, int32_t m,
                              void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(gate)) != TQ_OK) return st;
    if ((st = check_weight(up)) != TQ_OK) return st;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (up->n != gate->n || up->k != gate->k || up->fmt != gate->fmt) return TQ_ERR_INVALID_ARG;
    const int hidden = gate->k, inter = gate->n;
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    if ((st = check_smem(gate->fmt, m, true, gate->k, gate->n)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    return cuda_status(launch_gateup(gate, up, P.qx, P.sx, m, P.h, P.qh, P.sh, P.counters, P.err,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_ffn_stage_down(const tq_weight *down, int32_t m, float *y, void *workspace,
                            size_t workspace_bytes, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(down)) != TQ_OK) return st;
    if (y == nullptr || m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (!aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    const int hidden = down->n, inter = down->k;
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    if ((st = check_smem(down->fmt, m, false, down->k, down->n)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    return cuda_status(launch_down(down, P.qh, P.sh, m, y, P.err, reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_ffn_step(const tq_weight *gate, const tq_weight *up, const tq_weight *down,
                      const uint16_t *x, int32_t m, float *y, void *workspace,
                      size_t workspace_bytes, tq_stream_t stream) {
    tq_status st = check_ffn(gate, up, down, m);
    if (st != TQ_OK) return st;
    if (x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    const int hidden = gate->k, inter = gate->n;
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    if ((st = check_ffn_smem(gate->fmt, m, hidden, inter)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (use_fused(gate->fmt, m, hidden, inter)) {
        tq::FfnFusedArgs f = fused_args(P, hidden, inter, 0.0f);
        f.num_layers = 1;
        f.x = x;
        f.y = y;
        set_layer(f, 0, gate, up, down);
        return cuda_status(tq::launch_ffn_fused(f, gate->fmt, m, s));
    }
    cudaError_t e = launch_rotq(x, m, hidden, P.qx, P.sx, s);
    if (e == cudaSuccess)
        e = launch_gateup(gate, up, P.qx, P.sx, m, P.h, P.qh, P.sh, P.counters, P.err, s);
    if (e == cudaSuccess) e = launch_down(down, P.qh, P.sh, m, y, P.err, s);
    return cuda_status(e);
}

tq_status tq_ffn_stack(const tq_weight *layers, int32_t num_layers, const uint16_t *x, int32_t m,
                       float eps, float *y, void *workspace, size_t workspace_bytes,
                       tq_stream_t stream) {
    if (layers == nullptr || num_layers < 1 || x == nullptr || y == nullptr)
        return TQ_ERR_INVALID_ARG;
    tq_status st;
    for (int l = 0; l < num_layers; ++l)
        if ((st = check_ffn(&layers[3 * l], &layers[3 * l + 1], &layers[3 * l + 2], m)) != TQ_OK)
            return st;
    const int hidden = layers[0].k, inter = layers[0].n;
    for (int l = 1; l < num_layers; ++l)
        if (layers[3 * l].k != hidden || layers[3 * l].n != inter) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    if ((st = check_ffn_smem(layers[0].fmt, m, hidden, inter)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (use_fused(layers[0].fmt, m, hidden, inter)) {
        // chunks of up to kFusedMaxLayers layers per launch; a chunk after the
        // first starts from the RMS-normalised output of the one before
        cudaError_t e = cudaSuccess;
        for (int l0 = 0; l0 < num_layers && e == cudaSuccess; l0 += tq::kFusedMaxLayers) {
            const int cnt = num_layers - l0 < tq::kFusedMaxLayers ? num_layers - l0 : tq::kFusedMaxLayers;
            tq::FfnFusedArgs f = fused_args(P, hidden, inter, eps);
            f.num_layers = cnt;
            f.input_is_y = l0 > 0;
            f.x = x;
            f.y_in = P.ybuf;
            f.y = l0 + cnt == num_layers ? y : P.ybuf;
            for (int i = 0; i < cnt; ++i)
                set_layer(f, i, &layers[3 * (l0 + i)], &layers[3 * (l0 + i) + 1], &layers[3 * (l0 + i) + 2]);
            e = tq::launch_ffn_fused(f, layers[0].fmt, m, s);
        }
        return cuda_status(e);
    }
    cudaError_t e = launch_rotq(x, m, hidden, P.qx, P.sx, s);
    for (int l = 0; l < num_layers && e == cudaSuccess; ++l) {
        const tq_weight *L = &layers[3 * l];
        if (l > 0)
            e = tq::launch_pdl(tq::rmsnorm_rotq_kernel, dim3(m), dim3(tq::kNormThreads), 0, s,
                               static_cast<const float *>(P.ybuf), hidden, eps, P.qx, P.sx,
                               static_cast<uint16_t *>(nullptr));
        if (e == cudaSuccess)
            e = launch_gateup(&L[0], &L[1], P.qx, P.sx, m, P.h, P.qh, P.sh, P.counters, P.err, s);
        if (e == cudaSuccess)
            e = launch_down(&L[2], P.qh, P.sh, m, l + 1 == num_layers ? y : P.ybuf, P.err, s);
    }
    return cuda_status(e);
}

tq_status tq_rmsnorm_bf16(const float *y, int32_t m, int32_t n, float eps, uint16_t *x_out,
                          tq_stream_t stream) {
    if (y == nullptr || x_out == nullptr || m < 1 || n < 1) return TQ_ERR_INVALID_ARG;
    return cuda_status(tq::launch_pdl(tq::rmsnorm_bf16_kernel, dim3(m), dim3(tq::kNormThreads), 0,
                                      reinterpret_cast<cudaStream_t>(stream), y, n, eps, x_out));
}

}  // extern "C"
