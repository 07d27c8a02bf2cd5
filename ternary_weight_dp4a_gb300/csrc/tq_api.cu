// tq_api.cu -- the C ABI of libtq (declared in include/tq.h): argument checks,
// workspace layout and kernel dispatch.  Every data pointer is a device
// pointer owned by the caller; nothing here allocates.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_kernel.cuh"
#include "tq_kernel_launch.h"
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
//   sync: u64 launch ticket, then u32 [inter/1024] per 1024-wide segment of h,
//   its rotated 128-blocks (both count up over every step kernel launched on
//   the workspace; tq_ffn_workspace_init zeroes them) |
//   hst i8 [m*inter] (h quantised again, staged as the down phase reads it:
//   per pass of rows r0.., [inter/128][rows][128] permuted) |
//   hsn (f32 scale, i32 0x4b400000 - sum q) [m][inter/128] |
//   hp f32 [m][inter] (h after the transform's first four butterfly stages,
//   per 128-block element e at 4 (e mod 32) + e / 32)
struct FfnWorkspace {
    size_t qx, sx, h, qh, sh, counters, ybuf, err, sync, hst, hsn, hp, total;
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
    w.sync = off; off = round_up(off + static_cast<size_t>(2 + (inter + 1023) / 1024) * 4, kWsAlign);
    w.hst = off; off = round_up(off + static_cast<size_t>(m * inter), kWsAlign);
    w.hsn = off; off = round_up(off + static_cast<size_t>(m * (inter / 128)) * 8, kWsAlign);
    w.hp = off;  off = round_up(off + static_cast<size_t>(m * inter) * 4, kWsAlign);
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
    unsigned long long *ticket;
    unsigned *segready;
    uint8_t *hst;
    float2 *hsn;
    float *hp;
};

FfnPtrs ffn_ptrs(void *ws, const FfnWorkspace &L) {
    uint8_t *b = static_cast<uint8_t *>(ws);
    return FfnPtrs{reinterpret_cast<int8_t *>(b + L.qx), reinterpret_cast<float *>(b + L.sx),
                   reinterpret_cast<uint16_t *>(b + L.h), reinterpret_cast<int8_t *>(b + L.qh),
                   reinterpret_cast<float *>(b + L.sh), reinterpret_cast<unsigned *>(b + L.counters),
                   reinterpret_cast<float *>(b + L.ybuf), reinterpret_cast<unsigned *>(b + L.err),
                   reinterpret_cast<unsigned long long *>(b + L.sync), reinterpret_cast<unsigned *>(b + L.sync) + 2, b + L.hst,
                   reinterpret_cast<float2 *>(b + L.hsn), reinterpret_cast<float *>(b + L.hp)};
}

tq_status check_weight(const tq_weight *w) {
    if (w == nullptr || w->codes == nullptr || w->scales == nullptr) return TQ_ERR_INVALID_ARG;
    if (w->n < 1 || w->k < 128 || w->k % 128 != 0) return TQ_ERR_INVALID_ARG;
    if (w->fmt != TQ_FMT_TERNARY2 && w->fmt != TQ_FMT_BINARY1) return TQ_ERR_INVALID_ARG;
    if (!aligned(w->codes, 32) || !aligned(w->scales, 2)) return TQ_ERR_ALIGNMENT;
    return TQ_OK;
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

tq_status check_ws(void *ws, size_t bytes, int m, int hidden, int inter) {
    if (ws == nullptr) return TQ_ERR_INVALID_ARG;
    if (!aligned(ws, kWsAlign)) return TQ_ERR_ALIGNMENT;
    if (bytes < ffn_layout(m, hidden, inter).total) return TQ_ERR_WORKSPACE;
    return TQ_OK;
}

cudaError_t launch_rotq(const uint16_t *x, int64_t m, int k, int8_t *q, float *s,
                        cudaStream_t stream) {
    const int64_t blocks = m * (k / 128);
    const int64_t warps_per_cta = 256 / 32;
    const unsigned grid = static_cast<unsigned>((blocks + warps_per_cta - 1) / warps_per_cta);
    return tq::launch_pdl(tq::rotate_quant_kernel, dim3(grid), dim3(256), 0, stream, x, blocks, k,
                          q, s);
}

tq::WeightRef wref(const tq_weight *w) {
    return tq::WeightRef{w->codes, w->scales, w->n, w->k};
}

// Packed rows run in passes of at most kMaxRowsPerPass rows; the arithmetic
// of a row does not depend on which rows share its pass.
int pass_rows(int m, int r0) {
    return m - r0 < tq::kMaxRowsPerPass ? m - r0 : tq::kMaxRowsPerPass;
}

// device limits last: every host-side check comes first
tq_status check_fits(const tq::Call &c) {
    cudaError_t e = cudaSuccess;
    const bool fits = tq::call_fits(c, &e);
    if (e != cudaSuccess) return cuda_status(e);
    return fits ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

tq::Call ffn_call(const tq_weight *gate, const tq_weight *up, const tq_weight *down, int fmt) {
    tq::Call c{};
    c.fmt = fmt;
    c.m = tq::kMaxRowsPerPass;
    if (gate != nullptr) {
        c.do_a = 1;
        c.wa[0] = wref(gate);
        c.wa[1] = wref(up);
    }
    if (down != nullptr) {
        c.do_b = 1;
        c.wb = wref(down);
    }
    return c;
}

// The workspace rows r0.. of an FFN call: every per-row array is [m][...]
void set_ws_rows(tq::Call &c, const FfnPtrs &P, int r0, int hidden, int inter) {
    c.qx = P.qx + static_cast<size_t>(r0) * hidden;
    c.sx = P.sx + static_cast<size_t>(r0) * (hidden / 128);
    c.h = P.h + static_cast<size_t>(r0) * inter;
    c.qh = P.qh + static_cast<size_t>(r0) * inter;
    c.sh = P.sh + static_cast<size_t>(r0) * (inter / 128);
    c.hst = P.hst + static_cast<size_t>(r0) * inter;
    c.hsn = P.hsn + static_cast<size_t>(r0) * (inter / 128);
    c.hp = P.hp + static_cast<size_t>(r0) * inter;
    c.hcount = P.counters;
    c.ticket = P.ticket;
    c.segready = P.segready;
    c.err = P.err;
}

}  // namespace

namespace tq {
// lets other translation units report through tq_last_cuda_error()
void record_cuda_error(int e) { g_last_cuda_error = e; }
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
    tq::Call c = ffn_call(nullptr, nullptr, w, w->fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const int nb = w->k / 128;
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        c.qb = q + static_cast<size_t>(r0) * w->k;
        c.sb = s + static_cast<size_t>(r0) * nb;
        c.y = y + static_cast<size_t>(r0) * w->n;
        c.dots = blockdots == nullptr ? nullptr : blockdots + static_cast<size_t>(r0) * w->n * nb;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
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
    tq::Call c = ffn_call(gate, up, nullptr, gate->fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const int hidden = gate->k, inter = gate->n;
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    c.in_mode = tq::kInPlain;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        c.qa = qx + static_cast<size_t>(r0) * hidden;
        c.sa = sx + static_cast<size_t>(r0) * (hidden / 128);
        c.h = h + static_cast<size_t>(r0) * inter;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
}

size_t tq_ffn_workspace_bytes(int32_t m, int32_t hidden, int32_t inter) {
    if (m < 1 || hidden < 1 || inter < 1) return 0;
    return ffn_layout(m, hidden, inter).total;
}

size_t tq_ffn_workspace_error_offset(int32_t m, int32_t hidden, int32_t inter) {
    if (m < 1 || hidden < 1 || inter < 1) return 0;
    return ffn_layout(m, hidden, inter).err;
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
    if (inter % 128 != 0) return TQ_ERR_INVALID_ARG;          // h is rotated per 128-block
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    tq::Call c = ffn_call(gate, up, nullptr, gate->fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    c.in_mode = tq::kInPlain;
    c.rotate_h = 1;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        set_ws_rows(c, P, r0, hidden, inter);
        c.qa = c.qx;
        c.sa = c.sx;
        c.qx = nullptr;
        c.sx = nullptr;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
}

tq_status tq_ffn_stage_down(const tq_weight *down, int32_t m, float *y, void *workspace,
                            size_t workspace_bytes, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(down)) != TQ_OK) return st;
    if (y == nullptr || m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (!aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    const int hidden = down->n, inter = down->k;
    if ((st = check_ws(workspace, workspace_bytes, m, hidden, inter)) != TQ_OK) return st;
    tq::Call c = ffn_call(nullptr, nullptr, down, down->fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        set_ws_rows(c, P, r0, hidden, inter);
        c.bst = c.hst;
        c.bsn = c.hsn;
        c.y = y + static_cast<size_t>(r0) * hidden;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
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
    tq::Call c = ffn_call(gate, up, down, gate->fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    c.in_mode = tq::kInRotX;
    c.rotate_h = 1;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        set_ws_rows(c, P, r0, hidden, inter);
        c.x = x + static_cast<size_t>(r0) * hidden;
        c.bst = c.hst;
        c.bsn = c.hsn;
        c.y = y + static_cast<size_t>(r0) * hidden;
        e = tq::launch_call(c, str);
    }
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
    tq::Call c = ffn_call(&layers[0], &layers[1], &layers[2], layers[0].fmt);
    if ((st = check_fits(c)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    c.rotate_h = 1;
    c.eps = eps;
    // rows are independent through the whole stack: each pass of rows runs
    // every layer; a layer after the first starts from the RMS-normalised
    // output of the one before (kept in ybuf, rewritten in place)
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0);
        set_ws_rows(c, P, r0, hidden, inter);
        float *ybuf = P.ybuf + static_cast<size_t>(r0) * hidden;
        for (int l = 0; l < num_layers && e == cudaSuccess; ++l) {
            c.wa[0] = wref(&layers[3 * l]);
            c.wa[1] = wref(&layers[3 * l + 1]);
            c.wb = wref(&layers[3 * l + 2]);
            c.in_mode = l == 0 ? tq::kInRotX : tq::kInNormY;
            c.x = x + static_cast<size_t>(r0) * hidden;
            c.y_in = ybuf;
            c.bst = c.hst;
            c.bsn = c.hsn;
            c.y = l + 1 == num_layers ? y + static_cast<size_t>(r0) * hidden : ybuf;
            e = tq::launch_call(c, str);
        }
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
