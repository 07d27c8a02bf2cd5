// tq_tc.h -- host interface of the tensor-core GEMV / FFN kernel
// (tq_tc_kernel.cuh): one launch runs phase A (gate/up), phase B (down or a
// plain GEMV), or both, for a pass of m <= 8 activation rows.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq_kernel_launch.h"

namespace tq {

struct TcCall {
    int fmt, m;                         // m in 1..8
    int do_a, do_b;
    WeightRef wa[2];                    // gate, up
    WeightRef wb;                       // down / the GEMV matrix
    int in_mode;                        // phase A input: rotate x, RMS-normalise y_in, plain qa/sa
    const uint16_t *x;
    const float *y_in;
    float eps;
    const int8_t *qa;
    const float *sa;
    int8_t *qx;                         // quantised input for the caller (may be null)
    float *sx;
    uint16_t *h;
    int rotate_h;
    int8_t *qh;
    float *sh;
    uint8_t *hst;                       // h as phase B's operand (written with qh)
    float2 *hsn;
    const uint8_t *bst;                 // phase B operand blocks + pairs
    const float2 *bsn;
    float *y;
    int32_t *dots;
    float *part_a, *part_b;             // segment sums
    unsigned *cnt_a, *cnt_b;            // per-tile unit counts (zero between launches)
    unsigned *segready;                 // per segment of h: blocks rotated (A+B launches)
    unsigned long long *ticket;         // launch tickets (A+B launches)
    unsigned *err;
};

// Bytes of a B operand for k columns (whole segments, 2 KB per 128-block,
// enough for any pass), of its (scale, sum q) pairs, and of the segment sums
// of an n x k matrix for a pass of up to 8 rows.
size_t tc_operand_bytes(int k);
size_t tc_pairs_bytes(int k);
size_t tc_partials_bytes(int n, int k);
int tc_tiles(int n);

// True when the tensor-core kernel can run this call on the current device
// (rows, segment counts and its shared-memory plan); *err gets any CUDA
// error from querying the device.
bool tc_applicable(const TcCall &c, cudaError_t *err);

cudaError_t tc_launch(const TcCall &c, cudaStream_t stream);

// Lay plain int8 rows q [m][k] (+ s [m][k/128]) out as a B operand.
cudaError_t tc_stage_operand(int fmt, int m, const int8_t *q, const float *s, int k, uint8_t *bst, float2 *bsn,
                             cudaStream_t stream);

}  // namespace tq
