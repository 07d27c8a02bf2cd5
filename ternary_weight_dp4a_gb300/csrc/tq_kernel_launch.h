// tq_kernel_launch.h -- host interface of the persistent GEMV / FFN kernel
// (tq_kernel.cuh): one launch runs phase A (gate/up), phase B (down or a
// plain GEMV), or both in one launch, for m <= 4 rows.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tq {

struct WeightRef {
    const uint8_t *codes;
    const uint16_t *scales;
    int n, k;
};

struct Call {
    int fmt, m;                         // m in 1..4
    int do_a, do_b;
    WeightRef wa[2];                    // gate, up
    WeightRef wb;                       // down / the GEMV matrix
    int in_mode;                        // kInRotX, kInNormY, kInPlain (phase A)
    const uint16_t *x;
    const float *y_in;
    float eps;
    const int8_t *qa;
    const float *sa;
    int8_t *qx;
    float *sx;
    uint16_t *h;
    int rotate_h;
    int8_t *qh;
    float *sh;
    uint8_t *hst;                       // h staged for phase B (written with qh)
    float2 *hsn;
    float *hp;                          // h after its first four butterfly stages (rotate_h)
    unsigned *hcount;
    const uint8_t *bst;                 // phase B input, staged; or plain qb/sb
    const float2 *bsn;
    const int8_t *qb;
    const float *sb;
    float *y;
    int32_t *dots;
    // phase-B-only launches: segment sums [tiles][segments][m][16] and unit
    // counts [tiles] (zero between launches) of 16-row tiles shared between
    // CTAs; null keeps whole tiles per CTA
    float *gpart;
    unsigned *gcnt;
    unsigned *segready;                 // per segment of h: rotated 128-blocks (A+B launches)
    unsigned long long *ticket;         // launch tickets (A+B launches)
    unsigned *err;
};

// True when the kernel's shared-memory plan for these sizes fits this device
// (*err receives any CUDA error from querying it).
bool call_fits(const Call &c, cudaError_t *err);

cudaError_t launch_call(const Call &c, cudaStream_t stream);

}  // namespace tq
