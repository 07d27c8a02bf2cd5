/*
 * tq.h -- C ABI of libtq, the GB300 (sm_103a) ternary-weight FFN decode library.
 *
 * The operation is the decode-time FFN of a ternary-weight model read "from
 * its stored ternary blocks ... through a dp4a GEMV with its int8 activation
 * staged in shared memory and produced by the Hadamard rotation", with
 * "packed steps of up to 8 rows ... each row bit-identical to its single-row
 * decode" (sparkinfer PR #1154, "decode and small packed batches read the FFN
 * from a ternary copy through a dp4a GEMV", Summary).
 *
 * Conventions for every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates no memory and keeps no device state between calls.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  No call synchronises the stream or the device.
 *   - Arrays are row-major and contiguous.  A call checks its arguments
 *     before launching anything; on an error nothing is launched and the
 *     outputs are untouched.
 *   - TQ_ERR_CUDA means a launch itself failed; tq_last_cuda_error() gives
 *     the cudaError_t of the most recent failure on the calling thread.
 *     Errors raised later by kernels in flight surface at the caller's next
 *     synchronisation, as for any CUDA call.
 *   - Outputs must not overlap inputs or each other.
 *   - Sizes: k and hidden/intermediate are multiples of 128; 1 <= m <= 64.
 *     Rows run in passes through one weight stream each: up to 8 rows per
 *     pass on the tensor-core kernel (the packed decode step is one pass), up
 *     to 4 on the dp4a kernel; 9..64 rows (verify or prefill blocks) run
 *     further passes, each re-reading the weights.
 *   - Two kernels implement every GEMV and FFN entry point and give
 *     identical bits: a dp4a kernel and a tensor-core kernel (weights decoded
 *     to e4m3 in tensor memory, tcgen05.mma against the int8 activation split
 *     into two exact e4m3 parts).  tq_set_engine chooses; the default uses the
 *     dp4a kernel, measured the faster on GB300 for the FFN step at every row
 *     count and for the GEMV on every measured shape except a long input
 *     (5120 x 17408) at 8 rows, wherever its shared-memory plan fits, and the
 *     tensor-core kernel elsewhere.
 *   - Floating point is IEEE binary32 with the rounding of each step
 *     documented at the entry point; results do not depend on m, on the
 *     stream or on how many SMs the GPU has.
 *
 * Weight layout (the pages fix none; this library fixes this one):
 *   TQ_FMT_TERNARY2: 2-bit codes, 4 per byte.  Weight j of row i is in byte
 *     i*(k/4) + j/4 at bits 2*(j%4)..2*(j%4)+1, least significant first;
 *     code 0 -> 0, 1 -> +1, 2 -> -1.  Code 3 must not occur (the kernels'
 *     result for it is unspecified).
 *   TQ_FMT_BINARY1: 1 bit per weight, 8 per byte.  Weight j of row i is bit
 *     j%8 of byte i*(k/8) + j/8; 1 -> +1, 0 -> -1.
 *   scales: one IEEE fp16 per 128-weight block per row, [n][k/128].
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *tq_stream_t;

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1, /* null pointer, size out of range, shape mismatch   */
    TQ_ERR_ALIGNMENT = 2,   /* a pointer lacks the alignment its argument needs */
    TQ_ERR_UNSUPPORTED = 3, /* valid but beyond this build's limits              */
    TQ_ERR_WORKSPACE = 4,   /* workspace smaller than tq_ffn_workspace_bytes()   */
    TQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed              */
    TQ_ERR_TIMEOUT = 6      /* a bounded wait inside a kernel ran out (reported
                               by tq_error_status / tq_read_error_word from a
                               workspace's error word; the call that launched
                               the kernel itself returned TQ_OK)                */
} tq_status;

typedef enum { TQ_FMT_TERNARY2 = 0, TQ_FMT_BINARY1 = 1 } tq_format;

/* One packed weight matrix W [n][k] in the layout above.
 * codes: 32-byte aligned.  scales: 2-byte aligned. */
typedef struct {
    const uint8_t *codes;
    const uint16_t *scales;
    int32_t n;
    int32_t k;
    int32_t fmt; /* tq_format */
} tq_weight;

/* Most activation rows in one call.  A pass of r = min(m, 4) rows also
 * needs about r * (k/128) * 152 bytes (156 for 1-bit) of shared memory per
 * CTA besides the weight ring, at most the device's opt-in limit (227 KB on
 * GB300); beyond it a call returns TQ_ERR_UNSUPPORTED. */
#define TQ_MAX_ROWS 64

/* Human-readable name of a status code (static string). */
const char *tq_status_string(tq_status s);

/* Kernel selection, process-wide (an atomic setting read at every call):
 * TQ_ENGINE_AUTO (default) uses the dp4a kernel where its plan fits and the
 * tensor-core kernel elsewhere; TQ_ENGINE_DP4A always the dp4a kernel;
 * TQ_ENGINE_TCGEN05 always the tensor-core kernel (a call it cannot serve
 * returns TQ_ERR_UNSUPPORTED).  Results do not depend on the engine. */
#define TQ_ENGINE_AUTO 0
#define TQ_ENGINE_DP4A 1
#define TQ_ENGINE_TCGEN05 2
tq_status tq_set_engine(int32_t engine);
int32_t tq_get_engine(void);

/* Status of an error word read back from a workspace: TQ_OK for 0, else
 * TQ_ERR_TIMEOUT (the bits say which wait ran out). */
tq_status tq_error_status(uint32_t error_word);

/* Read the error word at `error_word` (a device address inside a workspace)
 * after the work enqueued on `stream` so far: copies it to the host and
 * SYNCHRONISES the stream.  *value (may be NULL) receives the word; returns
 * tq_error_status(word), or TQ_ERR_CUDA if the copy failed. */
tq_status tq_read_error_word(const uint32_t *error_word, uint32_t *value, tq_stream_t stream);

/* Zero-fill any libtq workspace (an async memset on `stream`).  A workspace
 * must be zero-filled once before its first use; every call leaves it
 * reusable.  After a call that failed in flight (a CUDA error surfaced at
 * synchronisation, or an error word that is not zero), initialise it again. */
tq_status tq_workspace_init(void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* cudaError_t of the last failed CUDA call made by this library on the
 * calling thread (0 if none). */
int tq_last_cuda_error(void);

/* Pack weight codes into the layout above (a load-time step).
 * codes: uint8 [n][k]; for TQ_FMT_TERNARY2 each entry is 0, 1 or 2 (value
 * 0, +1, -1), for TQ_FMT_BINARY1 each entry is 0 or 1 (value -1, +1).  Only
 * the low 2 (resp. 1) bits of each entry are read.
 * packed: [n][k/4] or [n][k/8] bytes, 32-byte aligned. */
tq_status tq_pack_weights(const uint8_t *codes, int32_t n, int32_t k, int32_t fmt,
                          uint8_t *packed, tq_stream_t stream);

/* Rotate and quantise activations ("the Hadamard rotation emits that int8
 * copy", PR #1154 Summary).  For each row r and 128-block b of x (bf16 bits
 * [m][k]): v = H128 * x_block in fp32, computed as the fast transform's
 * butterflies for span 1, 2, 4, ..., 64 (a+b to the lower index, a-b to the
 * upper) followed by one multiply by (float)(1/sqrt(128)); then
 * s[r][b] = max|v| / 127 and q = round-half-even(v / s) clamped to
 * [-127, 127] (IEEE division); an all-zero block gives s = 0, q = 0.
 * q: int8 [m][k], 16-byte aligned.  s: fp32 [m][k/128].  x: 16-byte aligned.
 * 1 <= m <= 8 is not required here: any m >= 1. */
tq_status tq_rotate_quant(const uint16_t *x, int32_t m, int32_t k, int8_t *q, float *s,
                          tq_stream_t stream);

/* Bytes of the device workspace tq_gemv needs for an n x k matrix (any m). */
size_t tq_gemv_workspace_bytes(int32_t m, int32_t n, int32_t k);

/* Ternary/binary GEMV for a packed step of m rows (the "dp4a GEMV", PR #1154
 * Summary).  For row r and output i:
 *   d_b = sum_{j in block b} W[i][j] * q[r][j]          (exact int32)
 *   t_b = (float)d_b * (fp16->fp32(scales[i][b]) * s[r][b])
 *   S_j = (((0 + t_{8j}) + t_{8j+1}) + ...) + t_{min(8j+7, nb-1)}
 *                                       (fp32, segments of 8 consecutive blocks)
 *   y[r][i] = pairwise tree over S_0 .. S_{nseg-1}: each level adds nodes
 *             (0,1), (2,3), ... in order and passes an odd last node up,
 *             until one value remains,
 * which is the same for every m, so each row of a packed step is
 * bit-identical to its single-row result.
 * q: int8 [m][k] (16-byte aligned); s: fp32 [m][k/128]; y: fp32 [m][n].
 * blockdots: NULL, or int32 [m][n][k/128] receiving every d_b.
 * workspace: >= tq_gemv_workspace_bytes(m, n, k) bytes, 256-byte aligned,
 * zero-filled once by tq_workspace_init; its first 4 bytes are the error
 * word of the bounded waits (bits as for the FFN workspace, plus bit 5 the
 * tensor-core epilogue, bit 7 its fold queue, bit 8 its operand copies).
 * The workspace holds the input laid out for the tensor core and every
 * 128-row tile's segment sums (the tiles' 1024-wide segments are spread
 * over the SMs and folded by whichever CTA completes the tile).  Calls
 * sharing a workspace must not run concurrently. */
tq_status tq_gemv(const tq_weight *w, const int8_t *q, const float *s, int32_t m, float *y,
                  int32_t *blockdots, void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* The fused gate/up stage of the FFN step: for each row r and output i,
 *   g = gemv(gate, qx, sx)[r][i], u = gemv(up, qx, sx)[r][i]  (as tq_gemv)
 *   h[r][i] = bf16_rn(g / (1 + exp(-g)) * u)                   (as tq_ffn_step)
 * gate, up: [inter][hidden], same format; qx int8 [m][hidden] (16-byte
 * aligned); sx fp32 [m][hidden/128]; h: bf16 bits [m][inter].
 * workspace: an FFN workspace for (m, hidden, inter) (see below); its error
 * word reports a wait that ran out. */
tq_status tq_ffn_gateup(const tq_weight *gate, const tq_weight *up, const int8_t *qx,
                        const float *sx, int32_t m, uint16_t *h, void *workspace,
                        size_t workspace_bytes, tq_stream_t stream);

/* Bytes of device workspace tq_ffn_step / tq_ffn_stack need for these sizes. */
size_t tq_ffn_workspace_bytes(int32_t m, int32_t hidden, int32_t inter);

/* Byte offset in such a workspace of its error word (uint32, 4-byte aligned;
 * 0 for invalid sizes).  Every wait inside the FFN kernels is bounded (about
 * 0.5 s of GPU clock cycles); a wait that runs out ORs a bit into this word
 * and the kernel finishes without hanging, its outputs undefined:
 *   bit 0  the weight stream waited for a free ring slot
 *   bit 1  the weight stream waited for its last copies to land
 *   bit 2  a compute warp waited for a slot's weights
 *   bit 3  a compute warp waited for its unit to be issued
 *   bit 4  the weight stream waited for the input to be staged
 *   bit 6  the down phase waited for a 1024-wide segment of h to be rotated
 *   bit 5  (tensor-core kernel) the epilogue waited for an accumulator, the
 *          weight scales or the down phase's operand
 *   bit 7  (tensor-core kernel) the fold warps waited for a job
 *   bit 8  (tensor-core kernel) the down phase's operand copies at exit
 * (on the tensor-core kernel bits 0..3 name its weight stream, decoders and
 * MMA issue in the same order).  The word stays set until the workspace is
 * initialised again; tq_read_error_word reads it and returns TQ_ERR_TIMEOUT
 * when it is not zero. */
size_t tq_ffn_workspace_error_offset(int32_t m, int32_t hidden, int32_t inter);

/* tq_workspace_init under its earlier name. */
tq_status tq_ffn_workspace_init(void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* One decode FFN step for m packed rows:
 *   (qx, sx) = rotate_quant(x)                           [m][hidden]
 *   g = gemv(gate, qx, sx), u = gemv(up, qx, sx)         [m][inter]
 *   h = bf16_rn(g / (1 + exp(-g)) * u)                   [m][inter]
 *   (qh, sh) = rotate_quant(h);  y = gemv(down, qh, sh)  [m][hidden]
 * gate, up: [inter][hidden]; down: [hidden][inter]; all the same format.
 * exp(z) is computed as 2^n * P(r): n = round-half-even(z * log2 e),
 * r = fma(-n, L2, fma(-n, L1, z)) with L1 = ln 2 with its low 12 significand
 * bits cleared and L2 = ln 2 - L1, P the degree-7 Taylor polynomial by
 * Horner's rule with fused multiply-adds; z > 88.72283935546875 gives +inf,
 * z < -103.972084045410156 gives 0.  Division is IEEE.
 * x: bf16 bits [m][hidden], 16-byte aligned.  y: fp32 [m][hidden].
 * workspace: >= tq_ffn_workspace_bytes(m, hidden, inter) bytes, 256-byte
 * aligned, initialised once by tq_ffn_workspace_init; it holds the step's
 * intermediates (qx, sx, h, qh, sh, h quantised again in the layout the down
 * phase reads) and the step's synchronisation state: per 128-block of h a
 * count of published rows (every call leaves it at zero), a launch ticket
 * and per 1024-wide segment of h a count of rotated blocks (both count up
 * over the calls on the workspace; a launch derives its index from its
 * ticket).  After a call that failed in flight the workspace must be
 * initialised again.  Calls sharing a workspace must not run concurrently.
 * The step is one persistent launch per pass (at most 8 rows on the
 * tensor-core kernel, 4 on the dp4a kernel): every CTA first rotates and
 * quantises x into shared memory, then streams its share of gate/up; the CTA
 * that completes a 128-block of h rotates and quantises it, and the down
 * phase of each CTA starts on a segment of h as soon as that segment is
 * ready.  The launch uses programmatic stream serialisation, so it may start
 * while earlier work in the stream drains, reading nothing earlier work
 * writes until that work has completed. */
tq_status tq_ffn_step(const tq_weight *gate, const tq_weight *up, const tq_weight *down,
                      const uint16_t *x, int32_t m, float *y, void *workspace,
                      size_t workspace_bytes, tq_stream_t stream);

/* The three stages of tq_ffn_step as separate launches on the same workspace
 * (for timing a stage on its own): stage_input rotates and quantises x into
 * the workspace; stage_gateup runs gate/up + SiLU*up and the rotation of h;
 * stage_down writes y.  Issued in that order they compute tq_ffn_step. */
tq_status tq_ffn_stage_input(const uint16_t *x, int32_t m, int32_t hidden, int32_t inter,
                             void *workspace, size_t workspace_bytes, tq_stream_t stream);
tq_status tq_ffn_stage_gateup(const tq_weight *gate, const tq_weight *up, int32_t m,
                              void *workspace, size_t workspace_bytes, tq_stream_t stream);
tq_status tq_ffn_stage_down(const tq_weight *down, int32_t m, float *y, void *workspace,
                            size_t workspace_bytes, tq_stream_t stream);

/* A stack of num_layers FFN layers for m packed rows: layer 0 reads x (bf16
 * bits [m][hidden]); layer l > 0 reads rmsnorm_bf16(y_{l-1}, eps) (as
 * tq_rmsnorm_bf16); y (fp32 [m][hidden]) receives the last layer's output.
 * layers: 3 * num_layers weights, (gate, up, down) per layer, all of one
 * format and shape.  Workspace as for tq_ffn_step. */
tq_status tq_ffn_stack(const tq_weight *layers, int32_t num_layers, const uint16_t *x, int32_t m,
                       float eps, float *y, void *workspace, size_t workspace_bytes,
                       tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * FFN step without a caller-supplied workspace.  (The pages have no
 * counterpart to this entry point: it exists for callers, not for the method.)
 *
 * Some callers cannot allocate device memory at the point where they run the
 * step: a plugin inside a host application that owns every device allocation
 * and offers no allocator, or a real-time loop whose rules forbid calling the
 * allocator after start-up.  tq_ffn_step_static serves them: it computes
 * exactly what tq_ffn_step computes, with its scratch in a fixed array of
 * tq_ffn_static_workspace_bytes() bytes (about 2.5 MB) that is part of the
 * library.  Every GPU that loads the library holds one such array until the
 * process exits.  The call allocates nothing (no cudaMalloc, no cudaFree).
 *
 * Limits: m <= TQ_STATIC_MAX_ROWS, hidden <= TQ_STATIC_MAX_HIDDEN,
 * intermediate <= TQ_STATIC_MAX_INTER; larger sizes return
 * TQ_ERR_UNSUPPORTED before anything is launched.
 *
 * The step runs on the dp4a kernel (its part of the workspace is what the
 * array holds); the bits equal tq_ffn_step's on either engine.
 *
 * The first call on a device looks up the array's device address for that
 * device (cudaGetSymbolAddress) and keeps it for the life of the process, so
 * resetting the device (cudaDeviceReset) after that first call is not
 * supported; make that first call before beginning any stream capture.  Each call then zero-fills the part of the array it uses
 * with an asynchronous memset on `stream` before launching the step.
 * All calls on a device share the one array: calls whose work can overlap on
 * the GPU (different streams without ordering between them) race on it and
 * must not be issued. */
#define TQ_STATIC_MAX_ROWS 8
#define TQ_STATIC_MAX_HIDDEN 8192
#define TQ_STATIC_MAX_INTER 32768

size_t tq_ffn_static_workspace_bytes(void);

tq_status tq_ffn_step_static(const tq_weight *gate, const tq_weight *up, const tq_weight *down,
                             const uint16_t *x, int32_t m, float *y, tq_stream_t stream);

/* RMS-normalise (between stacked layers): for each row r,
 *   ss = sum_i y[r][i]^2 as 256 partial sums (partial t adds i = t, t+256, ...
 *        in ascending order from +0.0) combined pairwise at distance
 *        1, 2, 4, ..., 128;
 *   x_out[r][i] = bf16_rn(y[r][i] * (1 / sqrt(ss / n + eps)))
 * with IEEE sqrt and division.  y: fp32 [m][n]; x_out: bf16 bits [m][n]. */
tq_status tq_rmsnorm_bf16(const float *y, int32_t m, int32_t n, float eps, uint16_t *x_out,
                          tq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
