/*
 * tq_oracle.c -- plain, slow CPU oracle for the ternary-weight FFN decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant generator with
 * the CUDA library: every step below is written out from the method's
 * description, not from the kernels.
 *
 * What it computes (per decode token row r):
 *   1. x (bf16) is split into 128-element blocks, each block rotated by the
 *      normalised 128-point Walsh-Hadamard transform and quantised to int8
 *      with one fp32 absmax scale per block.  ("the Hadamard rotation emits
 *      that int8 copy for gate and up to share" -- sparkinfer PR #1154,
 *      "decode and small packed batches read the FFN from a ternary copy
 *      through a dp4a GEMV", Summary / commit message.)
 *   2. gate and up GEMVs over ternary weights: per output row n and block b
 *      an exact int32 dot of the int8 activation with the {-1,0,+1} weights,
 *      scaled by the block's fp16 weight scale and the activation block's
 *      fp32 scale, accumulated in fp32 in a fixed documented order
 *      (same PR: "dp4a GEMV"; "lane walk, per-block fold and shuffle tree").
 *   3. h = bf16(SiLU(gate) * up).
 *   4. h is rotated and quantised like x, then the down GEMV gives y (fp32).
 *   5. (stack only) x_next = bf16(RMS-normalise(y)).
 *   A packed step of m <= 8 rows is m independent copies of the above
 *   (same PR: "packed steps of up to 8 rows ... each row bit-identical to its
 *   single-row decode").
 *
 * The pages fix no byte layout, rounding mode, reduction order or exp; the
 * readings taken here are listed at each function.  Floating point is IEEE
 * binary32 exactly as written (build with -ffp-contract=off; fmaf only where
 * written).  Row loops may run on several OpenMP threads: that changes no
 * per-row arithmetic.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BLOCK 128

/* ------------------------------------------------------------------------- */
/* scalar format conversions                                                  */
/* ------------------------------------------------------------------------- */

static float bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 -> fp32: a bf16 is the top 16 bits of a binary32. */
float orc_bf16_to_f32(uint16_t b) { return bits_to_float((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even (the reading taken for every
 * "rounded to bf16" step).  NaN stays NaN. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u = float_to_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* IEEE binary16 -> fp32, decoded field by field (normals, subnormals, inf). */
float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (e == 0)       v = ldexp((double)mant, -24);           /* subnormal */
    else if (e == 31) v = mant ? NAN : INFINITY;
    else              v = ldexp((double)(mant | 0x400), e - 25);
    return (float)(sign ? -v : v);                             /* exact */
}

/* ------------------------------------------------------------------------- */
/* weight layout                                                              */
/* ------------------------------------------------------------------------- */
/* The pages fix no byte layout ("its stored ternary blocks", PR #1154
 * Summary; "one packed weight format", bonsai-edge-serve README, kernels/).
 * Reading taken:
 *   2-bit: code of weight k of row n in byte n*(k_dim/4) + k/4, bits
 *          2*(k%4)..2*(k%4)+1, least significant first; codes 0 -> 0,
 *          1 -> +1, 2 -> -1 (3 is never written; read back as 0).
 *   1-bit: bit k%8 of byte n*(k_dim/8) + k/8; bit 1 -> +1, bit 0 -> -1.
 *   scales: one fp16 per 128-weight block per row, [n][k_dim/128]. */

int8_t orc_code2_value(uint8_t c) { return c == 1 ? 1 : (c == 2 ? -1 : 0); }

void orc_pack2(const uint8_t *codes, int n, int k, uint8_t *packed) {
    for (int r = 0; r < n; r++)
        for (int j = 0; j < k / 4; j++) {
            uint8_t byte = 0;
            for (int t = 0; t < 4; t++)
                byte |= (uint8_t)((codes[(size_t)r * k + 4 * j + t] & 3u) << (2 * t));
            packed[(size_t)r * (k / 4) + j] = byte;
        }
}

void orc_unpack2(const uint8_t *packed, int n, int k, int8_t *w) {
    for (int r = 0; r < n; r++)
        for (int i = 0; i < k; i++) {
            uint8_t byte = packed[(size_t)r * (k / 4) + i / 4];
            w[(size_t)r * k + i] = orc_code2_value((byte >> (2 * (i % 4))) & 3u);
        }
}

void orc_pack1(const uint8_t *bits, int n, int k, uint8_t *packed) {
    for (int r = 0; r < n; r++)
        for (int j = 0; j < k / 8; j++) {
            uint8_t byte = 0;
            for (int t = 0; t < 8; t++)
                byte |= (uint8_t)((bits[(size_t)r * k + 8 * j + t] & 1u) << t);
            packed[(size_t)r * (k / 8) + j] = byte;
        }
}

void orc_unpack1(const uint8_t *packed, int n, int k, int8_t *w) {
    for (int r = 0; r < n; r++)
        for (int i = 0; i < k; i++) {
            uint8_t byte = packed[(size_t)r * (k / 8) + i / 8];
            w[(size_t)r * k + i] = ((byte >> (i % 8)) & 1u) ? 1 : -1;
        }
}

/* ------------------------------------------------------------------------- */
/* rotation + quantisation                                                    */
/* ------------------------------------------------------------------------- */

/* Normalised 128-point Walsh-Hadamard transform in natural (Sylvester) order,
 * H[i][j] = (-1)^popcount(i&j) / sqrt(128).  Reading taken for "the Hadamard
 * rotation" (PR #1154 Summary), which names neither the ordering nor the
 * arithmetic: the fast transform's in-place butterflies in fp32 for span
 * h = 1, 2, 4, ..., 64 (a+b to the lower index, a-b to the upper), then one
 * fp32 multiply by c = (float)(1/sqrt(128)). */
void orc_wht128(float *v) {
    for (int h = 1; h < ORC_BLOCK; h <<= 1)
        for (int i = 0; i < ORC_BLOCK; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    const float c = (float)(1.0 / sqrt(128.0));
    for (int i = 0; i < ORC_BLOCK; i++) v[i] = v[i] * c;
}

/* Symmetric absmax int8 quantisation of one rotated block (reading taken:
 * s = amax/127, q = round-half-even(v/s) clamped to [-127,127], IEEE
 * division; an all-zero block gives s = 0 and q = 0). */
void orc_quant_block(const float *v, int8_t *q, float *s) {
    float amax = 0.0f;
    for (int i = 0; i < ORC_BLOCK; i++) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        *s = 0.0f;
        for (int i = 0; i < ORC_BLOCK; i++) q[i] = 0;
        return;
    }
    float sc = amax / 127.0f;
    *s = sc;
    for (int i = 0; i < ORC_BLOCK; i++) {
        float t = rintf(v[i] / sc);
        if (t > 127.0f) t = 127.0f;
        if (t < -127.0f) t = -127.0f;
        q[i] = (int8_t)t;
    }
}

/* x: bf16 bits [m][k]; q: int8 [m][k]; s: fp32 [m][k/128]. Rows independent. */
void orc_rotate_quant(const uint16_t *x, int m, int k, int8_t *q, float *s) {
    int nb = k / ORC_BLOCK;
    for (int r = 0; r < m; r++)
        for (int b = 0; b < nb; b++) {
            float v[ORC_BLOCK];
            size_t off = (size_t)r * k + (size_t)b * ORC_BLOCK;
            for (int i = 0; i < ORC_BLOCK; i++) v[i] = orc_bf16_to_f32(x[off + i]);
            orc_wht128(v);
            orc_quant_block(v, q + off, s + (size_t)r * nb + b);
        }
}

/* ------------------------------------------------------------------------- */
/* ternary / binary GEMV                                                      */
/* ------------------------------------------------------------------------- */

static int8_t weight_at(const uint8_t *packed, int fmt, int k, int n, int i) {
    if (fmt == 0) {
        uint8_t byte = packed[(size_t)n * (k / 4) + i / 4];
        return orc_code2_value((byte >> (2 * (i % 4))) & 3u);
    }
    uint8_t byte = packed[(size_t)n * (k / 8) + i / 8];
    return ((byte >> (i % 8)) & 1u) ? 1 : -1;
}

/* Exact int32 block dot of weight row n, block b with activation row q. */
static int32_t block_dot(const uint8_t *packed, int fmt, int k, int n, int b,
                         const int8_t *qrow) {
    int32_t acc = 0;
    for (int i = b * ORC_BLOCK; i < (b + 1) * ORC_BLOCK; i++)
        acc += (int32_t)weight_at(packed, fmt, k, n, i) * (int32_t)qrow[i];
    return acc;
}

/* dots: int32 [m][n][k/128]. */
void orc_blockdots(const uint8_t *packed, int fmt, int n, int k,
                   const int8_t *q, int m, int32_t *dots) {
    int nb = k / ORC_BLOCK;
    for (int r = 0; r < m; r++) {
#pragma omp parallel for schedule(static)
        for (int row = 0; row < n; row++)
            for (int b = 0; b < nb; b++)
                dots[((size_t)r * n + row) * nb + b] =
                    block_dot(packed, fmt, k, row, b, q + (size_t)r * k);
    }
}

/* The documented fp32 fold and reduction of one output.
 * Per block: t_b = (float)dot_b * (fp32(sw[n,b]) * s[r,b])  (two roundings,
 * that association).  Lane walk: the blocks split into segments of eight
 * consecutive blocks (the last one shorter when nb is not a multiple of 8);
 * segment j adds t_b for b = 8j, 8j+1, ... in ascending order starting from
 * +0.0f.  Shuffle tree: the segment sums combine pairwise, level by level --
 * node i of the next level is left + right of nodes 2i and 2i+1, and an odd
 * last node passes up unchanged -- until one value remains.
 * Reading taken for "each row's lane walk, per-block fold and shuffle tree"
 * (PR #1154 commit message): the pages fix no lane count or block order, so
 * the walk is taken over consecutive blocks; the order does not depend on
 * how many rows share the step. */
#define ORC_SEG 8
static float fold_output(const int32_t *dots_nb, const uint16_t *sw_row,
                         const float *s_row, int nb) {
    int nseg = (nb + ORC_SEG - 1) / ORC_SEG;
    float *node = (float *)malloc(sizeof(float) * (size_t)nseg);
    for (int j = 0; j < nseg; j++) {
        float acc = 0.0f;
        for (int b = j * ORC_SEG; b < nb && b < (j + 1) * ORC_SEG; b++) {
            float ws = orc_f16_to_f32(sw_row[b]) * s_row[b];
            float t = (float)dots_nb[b] * ws;
            acc = acc + t;
        }
        node[j] = acc;
    }
    int cnt = nseg;
    while (cnt > 1) {
        int next = 0;
        for (int i = 0; i + 1 < cnt; i += 2) node[next++] = node[i] + node[i + 1];
        if (cnt % 2 == 1) node[next++] = node[cnt - 1];
        cnt = next;
    }
    float y = node[0];
    free(node);
    return y;
}

/* y: fp32 [m][n].  scales: fp16 bits [n][k/128]. */
void orc_gemv(const uint8_t *packed, const uint16_t *scales, int fmt, int n, int k,
              const int8_t *q, const float *s, int m, float *y) {
    int nb = k / ORC_BLOCK;
    for (int r = 0; r < m; r++) {
        const int8_t *qrow = q + (size_t)r * k;
        const float *srow = s + (size_t)r * nb;
#pragma omp parallel for schedule(static)
        for (int row = 0; row < n; row++) {
            int32_t dots[ORC_BLOCK * 8];  /* k <= 131072 */
            int32_t *d = nb <= ORC_BLOCK * 8 ? dots : (int32_t *)malloc(sizeof(int32_t) * nb);
            for (int b = 0; b < nb; b++) d[b] = block_dot(packed, fmt, k, row, b, qrow);
            y[(size_t)r * n + row] = fold_output(d, scales + (size_t)row * nb, srow, nb);
            if (d != dots) free(d);
        }
    }
}

/* The plain definition in fp64: y = sum over blocks, in block order, of
 * dot_b * sw[n,b] * s[r,b].  Used for the relative-error bound. */
void orc_gemv_f64(const uint8_t *packed, const uint16_t *scales, int fmt, int n, int k,
                  const int8_t *q, const float *s, int m, double *y) {
    int nb = k / ORC_BLOCK;
    for (int r = 0; r < m; r++) {
#pragma omp parallel for schedule(static)
        for (int row = 0; row < n; row++) {
            double acc = 0.0;
            for (int b = 0; b < nb; b++) {
                int32_t d = block_dot(packed, fmt, k, row, b, q + (size_t)r * k);
                acc += (double)d * (double)orc_f16_to_f32(scales[(size_t)row * nb + b]) *
                       (double)s[(size_t)r * nb + b];
            }
            y[(size_t)r * n + row] = acc;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* SiLU(gate) * up                                                            */
/* ------------------------------------------------------------------------- */

/* exp(x) in binary32 by Cody-Waite range reduction and a Taylor polynomial
 * (W. J. Cody and W. Waite, "Software Manual for the Elementary Functions",
 * 1980, chapter on exp): x = n*ln2 + r with n = round-half-even(x*log2(e)),
 * r = (x - n*L1) - n*L2 evaluated with fmaf, where L1 is ln2 with its low 12
 * significand bits cleared and L2 = ln2 - L1; exp(r) = sum_{j<=7} r^j/j!
 * by Horner's rule with fmaf; the result is scaled by 2^n as two exact
 * power-of-two multiplies.  Written out here so that both sides of the
 * parity check round identically (the pages name no exp). */
float orc_expf(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return INFINITY;
    if (x < -103.972084045410156f) return 0.0f;
    const double ln2 = 0.69314718055994530942;
    const float L1 = bits_to_float(float_to_bits((float)ln2) & 0xfffff000u);
    const float L2 = (float)(ln2 - (double)L1);
    const float log2e = (float)1.44269504088896340736;
    float n = rintf(x * log2e);
    float r = fmaf(-n, L1, x);
    r = fmaf(-n, L2, r);
    /* Horner: 1 + r(1 + r(1/2 + r(1/6 + ... r/5040))) */
    static const double inv_fact[8] = {1.0, 1.0, 1.0 / 2, 1.0 / 6, 1.0 / 24, 1.0 / 120,
                                       1.0 / 720, 1.0 / 5040};
    float p = (float)inv_fact[7];
    for (int j = 6; j >= 0; j--) p = fmaf(p, r, (float)inv_fact[j]);
    int ni = (int)n;
    int n1 = ni / 2, n2 = ni - n1;
    float s1 = bits_to_float((uint32_t)(n1 + 127) << 23);
    float s2 = bits_to_float((uint32_t)(n2 + 127) << 23);
    return (p * s1) * s2;
}

/* SiLU(g) = g / (1 + exp(-g)) in fp32 with IEEE division. */
float orc_silu(float g) { return g / (1.0f + orc_expf(-g)); }

/* h = bf16_rn(SiLU(g) * u) elementwise. */
void orc_silu_mul_bf16(const float *g, const float *u, size_t count, uint16_t *h) {
    for (size_t i = 0; i < count; i++) h[i] = orc_f32_to_bf16(orc_silu(g[i]) * u[i]);
}

/* ------------------------------------------------------------------------- */
/* FFN step                                                                   */
/* ------------------------------------------------------------------------- */

/* One decode FFN step for m rows: rotate+quant(x) -> gate, up -> bf16(SiLU(g)*u)
 * -> rotate+quant(h) -> down.  Reading taken: the down GEMV's input is h
 * rounded to bf16 and rotated/quantised exactly like x (the weights are taken
 * as stored in the rotated basis; no inverse rotation is applied).
 * Every intermediate buffer may be NULL except y. */
void orc_ffn_step(const uint8_t *gate, const uint16_t *gate_s,
                  const uint8_t *up, const uint16_t *up_s,
                  const uint8_t *down, const uint16_t *down_s, int fmt,
                  int hidden, int inter, const uint16_t *x, int m, float *y,
                  int8_t *qx_out, float *sx_out, float *g_out, float *u_out,
                  uint16_t *h_out, int8_t *qh_out, float *sh_out) {
    size_t mh = (size_t)m * hidden, mi = (size_t)m * inter;
    int8_t *qx = (int8_t *)malloc(mh);
    float *sx = (float *)malloc(sizeof(float) * (mh / ORC_BLOCK));
    float *g = (float *)malloc(sizeof(float) * mi);
    float *u = (float *)malloc(sizeof(float) * mi);
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * mi);
    int8_t *qh = (int8_t *)malloc(mi);
    float *sh = (float *)malloc(sizeof(float) * (mi / ORC_BLOCK));

    orc_rotate_quant(x, m, hidden, qx, sx);
    orc_gemv(gate, gate_s, fmt, inter, hidden, qx, sx, m, g);
    orc_gemv(up, up_s, fmt, inter, hidden, qx, sx, m, u);
    orc_silu_mul_bf16(g, u, mi, h);
    orc_rotate_quant(h, m, inter, qh, sh);
    orc_gemv(down, down_s, fmt, hidden, inter, qh, sh, m, y);

    if (qx_out) memcpy(qx_out, qx, mh);
    if (sx_out) memcpy(sx_out, sx, sizeof(float) * (mh / ORC_BLOCK));
    if (g_out) memcpy(g_out, g, sizeof(float) * mi);
    if (u_out) memcpy(u_out, u, sizeof(float) * mi);
    if (h_out) memcpy(h_out, h, sizeof(uint16_t) * mi);
    if (qh_out) memcpy(qh_out, qh, mi);
    if (sh_out) memcpy(sh_out, sh, sizeof(float) * (mi / ORC_BLOCK));
    free(qx); free(sx); free(g); free(u); free(h); free(qh); free(sh);
}

/* ------------------------------------------------------------------------- */
/* RMS-normalise (layer stack)                                                */
/* ------------------------------------------------------------------------- */

/* x_out = bf16_rn(y * (1 / sqrt(mean(y^2) + eps))), no gain.  Reading taken
 * (the stack's "RMS-normalise" names no gain, eps or order): the sum of
 * squares is 256 partial sums, partial t adding y[i]*y[i] for
 * i = t, t+256, ... in ascending order from +0.0f, combined pairwise at
 * distance 1, 2, 4, ..., 128; mean = sum / n; 1/sqrt with IEEE sqrt and
 * division. */
void orc_rmsnorm_bf16(const float *y, int m, int n, float eps, uint16_t *x_out) {
    for (int r = 0; r < m; r++) {
        const float *yr = y + (size_t)r * n;
        float part[256];
        for (int t = 0; t < 256; t++) {
            float acc = 0.0f;
            for (int i = t; i < n; i += 256) acc = acc + yr[i] * yr[i];
            part[t] = acc;
        }
        for (int d = 1; d < 256; d <<= 1)
            for (int t = 0; t < 256; t++)
                if ((t & d) == 0 && (t & (2 * d - 1)) == 0) part[t] = part[t] + part[t + d];
        float ms = part[0] / (float)n;
        float inv = 1.0f / sqrtf(ms + eps);
        for (int i = 0; i < n; i++) x_out[(size_t)r * n + i] = orc_f32_to_bf16(yr[i] * inv);
    }
}

/* ------------------------------------------------------------------------- */

void orc_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
