// tq_api.cu -- the C ABI of libtq (declared in include/tq.h): argument checks,
// workspace layout and kernel dispatch.  Every data pointer is a device
// pointer owned by the caller; nothing here allocates.
//
// Two kernels compute every GEMV and FFN entry point with identical results:
// the dp4a kernel (tq_kernel.cuh) and the tensor-core kernel
// (tq_tc_kernel.cuh, passes of up to 8 rows).  The engine setting picks one;
// the default takes the dp4a kernel (the faster, measured) wherever its
// shared-memory plan fits.
#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_kernel.cuh"
#include "tq_kernel_launch.h"
#include "tq_launch.h"
#include "tq_misc.cuh"
#include "tq_norm_kernels.cuh"
#include "tq_tc.h"
#include "tq_workspace.h"

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_engine{TQ_ENGINE_AUTO};

tq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    g_last_cuda_error = static_cast<int>(e);
    return TQ_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using tq::FfnWorkspace;
using tq::ffn_layout;
using tq::gemv_layout;
using tq::GemvWorkspace;
using tq::kWsAlign;

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
    uint8_t *tc_hst;
    float2 *tc_hsn;
    float *part_a, *part_b;
    unsigned *cnt_a, *cnt_b;
    float *ybuf2;
};

FfnPtrs ffn_ptrs(void *ws, const FfnWorkspace &L) {
    uint8_t *b = static_cast<uint8_t *>(ws);
    FfnPtrs p{};
    p.qx = reinterpret_cast<int8_t *>(b + L.qx);
    p.sx = reinterpret_cast<float *>(b + L.sx);
    p.h = reinterpret_cast<uint16_t *>(b + L.h);
    p.qh = reinterpret_cast<int8_t *>(b + L.qh);
    p.sh = reinterpret_cast<float *>(b + L.sh);
    p.counters = reinterpret_cast<unsigned *>(b + L.counters);
    p.ybuf = reinterpret_cast<float *>(b + L.ybuf);
    p.err = reinterpret_cast<unsigned *>(b + L.err);
    p.ticket = reinterpret_cast<unsigned long long *>(b + L.sync);
    p.segready = reinterpret_cast<unsigned *>(b + L.sync) + 2;
    p.hst = b + L.hst;
    p.hsn = reinterpret_cast<float2 *>(b + L.hsn);
    p.hp = reinterpret_cast<float *>(b + L.hp);
    p.tc_hst = b + L.tc_hst;
    p.tc_hsn = reinterpret_cast<float2 *>(b + L.tc_hsn);
    p.part_a = reinterpret_cast<float *>(b + L.part_a);
    p.part_b = reinterpret_cast<float *>(b + L.part_b);
    p.cnt_a = reinterpret_cast<unsigned *>(b + L.cnt_a);
    p.cnt_b = reinterpret_cast<unsigned *>(b + L.cnt_b);
    p.ybuf2 = reinterpret_cast<float *>(b + L.ybuf2);
    return p;
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

tq_status check_ws(void *ws, size_t bytes, size_t need) {
    if (ws == nullptr) return TQ_ERR_INVALID_ARG;
    if (!aligned(ws, kWsAlign)) return TQ_ERR_ALIGNMENT;
    if (bytes < need) return TQ_ERR_WORKSPACE;
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

// Rows run in passes; the arithmetic of a row does not depend on which rows
// share its pass.  The tensor-core kernel takes up to 8 rows per pass, the
// dp4a kernel up to 4.
constexpr int kTcPass = 8;

int pass_rows(int m, int r0, int per) { return m - r0 < per ? m - r0 : per; }

// ---- engine choice -----------------------------------------------------------
// TQ_ENGINE_AUTO takes the dp4a kernel: measured on GB300 it is the faster of
// the two at every row count (a tcgen05.mma of M = 128, K = 32 costs ~145
// cycles whatever N is, so the tensor-core kernel cannot stream the weights
// faster than ~30 us per 71 MB FFN layer, and its pipeline's latencies add
// to that), and the tensor-core kernel only where the dp4a kernel's plan
// does not fit.  The tensor-core kernel's plan for a pass of min(m, 8) rows
// decides for the whole call (a smaller last pass needs less).  Returns TQ_OK
// with *tc set, or an error (TQ_ERR_UNSUPPORTED when the tensor-core engine
// is forced and does not fit, TQ_ERR_CUDA when a device query fails).
tq_status choose_engine(tq::TcCall c, int m, bool *tc, const tq::Call *dp4a_fallback = nullptr) {
    const int engine = g_engine.load();
    *tc = false;
    if (engine == TQ_ENGINE_DP4A) return TQ_OK;
    cudaError_t e = cudaSuccess;
    if (engine == TQ_ENGINE_AUTO) {
        if (dp4a_fallback == nullptr) return TQ_OK;
        const bool dp4a_fits = tq::call_fits(*dp4a_fallback, &e);
        if (e != cudaSuccess) return cuda_status(e);
        if (dp4a_fits) return TQ_OK;
    }
    c.m = m < kTcPass ? m : kTcPass;
    const bool ok = tq::tc_applicable(c, &e);
    if (e != cudaSuccess) return cuda_status(e);
    if (!ok && engine == TQ_ENGINE_TCGEN05) return TQ_ERR_UNSUPPORTED;
    *tc = ok;
    return TQ_OK;
}

// device limits last: every host-side check comes first
tq_status check_fits_dp4a(const tq::Call &c) {
    cudaError_t e = cudaSuccess;
    const bool fits = tq::call_fits(c, &e);
    if (e != cudaSuccess) return cuda_status(e);
    return fits ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

// A phase-B-only dp4a call shares tiles between CTAs (equal shares of the
// units) through the workspace's segment sums and per-tile counts, when its
// plan fits with them; otherwise it deals whole tiles.
void share_tiles(tq::Call &c, float *gpart, unsigned *gcnt) {
    c.gpart = gpart;
    c.gcnt = gcnt;
    cudaError_t e = cudaSuccess;
    if (!tq::call_fits(c, &e)) {
        c.gpart = nullptr;
        c.gcnt = nullptr;
    }
}

tq::Call dp4a_call(const tq_weight *gate, const tq_weight *up, const tq_weight *down, int fmt) {
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

tq::TcCall tc_call(const tq_weight *gate, const tq_weight *up, const tq_weight *down, int fmt) {
    tq::TcCall c{};
    c.fmt = fmt;
    c.m = kTcPass;
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

// The workspace rows r0.. of a dp4a FFN call: every per-row array is [m][...]
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

// The workspace rows r0.. of a tensor-core FFN call; the operand copy of h
// and its pairs are per pass (r0 / 8), the segment sums and counts shared.
void set_tc_rows(tq::TcCall &c, const FfnPtrs &P, int r0, int hidden, int inter) {
    c.qx = P.qx + static_cast<size_t>(r0) * hidden;
    c.sx = P.sx + static_cast<size_t>(r0) * (hidden / 128);
    c.h = P.h + static_cast<size_t>(r0) * inter;
    c.qh = P.qh + static_cast<size_t>(r0) * inter;
    c.sh = P.sh + static_cast<size_t>(r0) * (inter / 128);
    c.hst = P.tc_hst + static_cast<size_t>(r0 / kTcPass) * tq::tc_ws_operand(inter);
    c.hsn = reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(P.tc_hsn) +
                                       static_cast<size_t>(r0 / kTcPass) * tq::tc_ws_pairs(inter));
    c.bst = c.hst;
    c.bsn = c.hsn;
    c.part_a = P.part_a;
    c.part_b = P.part_b;
    c.cnt_a = P.cnt_a;
    c.cnt_b = P.cnt_b;
    c.segready = P.segready;
    c.ticket = P.ticket;
    c.err = P.err;
}

}  // namespace

namespace tq {
// lets other translation units report through tq_last_cuda_error()
void record_cuda_error(int e) { g_last_cuda_error = e; }

// The FFN step on the dp4a kernel alone (the no-allocation entry point uses
// it: its built-in scratch holds the dp4a kernel's part of the workspace).
tq_status ffn_step_dp4a(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                        int32_t m, float *y, void *workspace, cudaStream_t str);
tq_status ffn_check_args(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                         int32_t m, const float *y);
}  // namespace tq

tq_status tq::ffn_check_args(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                             int32_t m, const float *y) {
    tq_status st = check_ffn(gate, up, down, m);
    if (st != TQ_OK) return st;
    if (x == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    return TQ_OK;
}

tq_status tq::ffn_step_dp4a(const tq_weight *gate, const tq_weight *up, const tq_weight *down, const uint16_t *x,
                            int32_t m, float *y, void *workspace, cudaStream_t str) {
    const int hidden = gate->k, inter = gate->n;
    tq::Call c = dp4a_call(gate, up, down, gate->fmt);
    tq_status st;
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, ffn_layout(m, hidden, inter));
    cudaError_t e = cudaSuccess;
    c.in_mode = tq::kInRotX;
    c.rotate_h = 1;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
        set_ws_rows(c, P, r0, hidden, inter);
        c.x = x + static_cast<size_t>(r0) * hidden;
        c.bst = c.hst;
        c.bsn = c.hsn;
        c.y = y + static_cast<size_t>(r0) * hidden;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
}

extern "C" {

const char *tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_ALIGNMENT: return "misaligned pointer";
        case TQ_ERR_UNSUPPORTED: return "unsupported size";
        case TQ_ERR_WORKSPACE: return "workspace too small";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    }
    return "unknown status";
}

int tq_last_cuda_error(void) { return g_last_cuda_error; }

tq_status tq_set_engine(int32_t engine) {
    if (engine != TQ_ENGINE_AUTO && engine != TQ_ENGINE_DP4A && engine != TQ_ENGINE_TCGEN05)
        return TQ_ERR_INVALID_ARG;
    g_engine.store(engine);
    return TQ_OK;
}

int32_t tq_get_engine(void) { return g_engine.load(); }

tq_status tq_error_status(uint32_t error_word) { return error_word == 0u ? TQ_OK : TQ_ERR_TIMEOUT; }

tq_status tq_read_error_word(const uint32_t *error_word, uint32_t *value, tq_stream_t stream) {
    if (error_word == nullptr) return TQ_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, error_word, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    if (value != nullptr) *value = v;
    return tq_error_status(v);
}

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

size_t tq_gemv_workspace_bytes(int32_t m, int32_t n, int32_t k) {
    if (m < 1 || n < 1 || k < 128) return 0;
    return gemv_layout(n, k).total;
}

tq_status tq_workspace_init(void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (workspace == nullptr) return TQ_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_gemv(const tq_weight *w, const int8_t *q, const float *s, int32_t m, float *y,
                  int32_t *blockdots, void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    tq_status st = check_weight(w);
    if (st != TQ_OK) return st;
    if (q == nullptr || s == nullptr || y == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(s, 4) || !aligned(y, 4) || !aligned(blockdots, 4))
        return TQ_ERR_ALIGNMENT;
    const GemvWorkspace L = gemv_layout(w->n, w->k);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    unsigned *err = reinterpret_cast<unsigned *>(wsb + L.err);
    const int nb = w->k / 128;
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    tq::TcCall tc = tc_call(nullptr, nullptr, w, w->fmt);
    const tq::Call dpc = dp4a_call(nullptr, nullptr, w, w->fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    if (use_tc) {
        uint8_t *bst = wsb + L.operand;
        float2 *bsn = reinterpret_cast<float2 *>(wsb + L.pairs);
        tc.bst = bst;
        tc.bsn = bsn;
        tc.part_b = reinterpret_cast<float *>(wsb + L.part);
        tc.cnt_b = reinterpret_cast<unsigned *>(wsb + L.cnt);
        tc.err = err;
        for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
            tc.m = pass_rows(m, r0, kTcPass);
            const int8_t *qp = q + static_cast<size_t>(r0) * w->k;
            const float *sp = s + static_cast<size_t>(r0) * nb;
            e = tq::tc_stage_operand(w->fmt, tc.m, qp, sp, w->k, bst, bsn, str);
            if (e != cudaSuccess) break;
            tc.y = y + static_cast<size_t>(r0) * w->n;
            tc.dots = blockdots == nullptr ? nullptr : blockdots + static_cast<size_t>(r0) * w->n * nb;
            e = tq::tc_launch(tc, str);
        }
        return cuda_status(e);
    }
    tq::Call c = dp4a_call(nullptr, nullptr, w, w->fmt);
    share_tiles(c, reinterpret_cast<float *>(wsb + L.part), reinterpret_cast<unsigned *>(wsb + L.cnt));
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    c.err = err;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
        c.qb = q + static_cast<size_t>(r0) * w->k;
        c.sb = s + static_cast<size_t>(r0) * nb;
        c.y = y + static_cast<size_t>(r0) * w->n;
        c.dots = blockdots == nullptr ? nullptr : blockdots + static_cast<size_t>(r0) * w->n * nb;
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
    return tq_workspace_init(workspace, workspace_bytes, stream);
}

tq_status tq_ffn_gateup(const tq_weight *gate, const tq_weight *up, const int8_t *qx,
                        const float *sx, int32_t m, uint16_t *h, void *workspace,
                        size_t workspace_bytes, tq_stream_t stream) {
    tq_status st;
    if ((st = check_weight(gate)) != TQ_OK) return st;
    if ((st = check_weight(up)) != TQ_OK) return st;
    if (qx == nullptr || sx == nullptr || h == nullptr) return TQ_ERR_INVALID_ARG;
    if (m < 1 || m > TQ_MAX_ROWS) return TQ_ERR_INVALID_ARG;
    if (up->n != gate->n || up->k != gate->k || up->fmt != gate->fmt) return TQ_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(sx, 4) || !aligned(h, 2)) return TQ_ERR_ALIGNMENT;
    const int hidden = gate->k, inter = gate->n;
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, L);
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    tq::TcCall tc = tc_call(gate, up, nullptr, gate->fmt);
    const tq::Call dpc = dp4a_call(gate, up, nullptr, gate->fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    if (use_tc) {
        tc.in_mode = tq::kInPlain;
        tc.part_a = P.part_a;
        tc.cnt_a = P.cnt_a;
        tc.err = P.err;
        for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
            tc.m = pass_rows(m, r0, kTcPass);
            tc.qa = qx + static_cast<size_t>(r0) * hidden;
            tc.sa = sx + static_cast<size_t>(r0) * (hidden / 128);
            tc.h = h + static_cast<size_t>(r0) * inter;
            e = tq::tc_launch(tc, str);
        }
        return cuda_status(e);
    }
    tq::Call c = dp4a_call(gate, up, nullptr, gate->fmt);
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    c.in_mode = tq::kInPlain;
    c.err = P.err;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
        c.qa = qx + static_cast<size_t>(r0) * hidden;
        c.sa = sx + static_cast<size_t>(r0) * (hidden / 128);
        c.h = h + static_cast<size_t>(r0) * inter;
        e = tq::launch_call(c, str);
    }
    return cuda_status(e);
}

tq_status tq_ffn_stage_input(const uint16_t *x, int32_t m, int32_t hidden, int32_t inter,
                             void *workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (x == nullptr || m < 1 || m > TQ_MAX_ROWS || hidden < 128 || hidden % 128 != 0 ||
        inter < 128 || inter % 128 != 0)
        return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16)) return TQ_ERR_ALIGNMENT;
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    tq_status st = check_ws(workspace, workspace_bytes, L.total);
    if (st != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, L);
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
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, L);
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    tq::TcCall tc = tc_call(gate, up, nullptr, gate->fmt);
    tc.rotate_h = 1;
    const tq::Call dpc = dp4a_call(gate, up, nullptr, gate->fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    if (use_tc) {
        tc.in_mode = tq::kInPlain;
        for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
            tc.m = pass_rows(m, r0, kTcPass);
            set_tc_rows(tc, P, r0, hidden, inter);
            tc.qa = tc.qx;
            tc.sa = tc.sx;
            tc.qx = nullptr;
            tc.sx = nullptr;
            e = tq::tc_launch(tc, str);
        }
        return cuda_status(e);
    }
    tq::Call c = dp4a_call(gate, up, nullptr, gate->fmt);
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    c.in_mode = tq::kInPlain;
    c.rotate_h = 1;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
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
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, L);
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    tq::TcCall tc = tc_call(nullptr, nullptr, down, down->fmt);
    const tq::Call dpc = dp4a_call(nullptr, nullptr, down, down->fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    if (use_tc) {
        for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
            tc.m = pass_rows(m, r0, kTcPass);
            set_tc_rows(tc, P, r0, hidden, inter);
            tc.y = y + static_cast<size_t>(r0) * hidden;
            e = tq::tc_launch(tc, str);
        }
        return cuda_status(e);
    }
    tq::Call c = dp4a_call(nullptr, nullptr, down, down->fmt);
    share_tiles(c, P.part_b, P.cnt_b);
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
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
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    tq::TcCall tc = tc_call(gate, up, down, gate->fmt);
    tc.rotate_h = 1;
    const tq::Call dpc = dp4a_call(gate, up, down, gate->fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    if (!use_tc) return tq::ffn_step_dp4a(gate, up, down, x, m, y, workspace, str);
    const FfnPtrs P = ffn_ptrs(workspace, L);
    cudaError_t e = cudaSuccess;
    tc.in_mode = tq::kInRotX;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
        tc.m = pass_rows(m, r0, kTcPass);
        set_tc_rows(tc, P, r0, hidden, inter);
        tc.x = x + static_cast<size_t>(r0) * hidden;
        tc.y = y + static_cast<size_t>(r0) * hidden;
        e = tq::tc_launch(tc, str);
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
        if (layers[3 * l].k != hidden || layers[3 * l].n != inter || layers[3 * l].fmt != layers[0].fmt)
            return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4)) return TQ_ERR_ALIGNMENT;
    const FfnWorkspace L = ffn_layout(m, hidden, inter);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != TQ_OK) return st;
    const FfnPtrs P = ffn_ptrs(workspace, L);
    cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    tq::TcCall tc = tc_call(&layers[0], &layers[1], &layers[2], layers[0].fmt);
    tc.rotate_h = 1;
    const tq::Call dpc = dp4a_call(&layers[0], &layers[1], &layers[2], layers[0].fmt);
    bool use_tc = false;
    if ((st = choose_engine(tc, m, &use_tc, &dpc)) != TQ_OK) return st;
    // rows are independent through the whole stack: each pass of rows runs
    // every layer; a layer after the first starts from the RMS-normalised
    // output of the one before
    if (use_tc) {
        tc.eps = eps;
        for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += kTcPass) {
            tc.m = pass_rows(m, r0, kTcPass);
            set_tc_rows(tc, P, r0, hidden, inter);
            // the layers alternate between two activation buffers, so no
            // launch reads the buffer it writes
            float *buf[2] = {P.ybuf + static_cast<size_t>(r0) * hidden, P.ybuf2 + static_cast<size_t>(r0) * hidden};
            for (int l = 0; l < num_layers && e == cudaSuccess; ++l) {
                tc.wa[0] = wref(&layers[3 * l]);
                tc.wa[1] = wref(&layers[3 * l + 1]);
                tc.wb = wref(&layers[3 * l + 2]);
                tc.in_mode = l == 0 ? tq::kInRotX : tq::kInNormY;
                tc.x = x + static_cast<size_t>(r0) * hidden;
                tc.y_in = buf[(l + 1) & 1];
                tc.y = l + 1 == num_layers ? y + static_cast<size_t>(r0) * hidden : buf[l & 1];
                e = tq::tc_launch(tc, str);
            }
        }
        return cuda_status(e);
    }
    tq::Call c = dp4a_call(&layers[0], &layers[1], &layers[2], layers[0].fmt);
    if ((st = check_fits_dp4a(c)) != TQ_OK) return st;
    c.rotate_h = 1;
    c.eps = eps;
    for (int r0 = 0; r0 < m && e == cudaSuccess; r0 += tq::kMaxRowsPerPass) {
        c.m = pass_rows(m, r0, tq::kMaxRowsPerPass);
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
