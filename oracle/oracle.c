/*
 * oracle.c -- the CPU oracle for the GGUF Q8_0 / Q4_0 decode DMMV.
 *
 * TEST INFRASTRUCTURE ONLY: only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this. Plain C99, no CUDA, no code shared
 * with the GPU library. Floating point that defines a result (the activation
 * quantizer) is done in fp32 exactly as the definition states; everything else
 * accumulates in fp64 in plain loop order so a reader can check it by eye.
 *
 * Definitions followed (page titles and sections; see oracle.h for the list):
 *  - DMMV = dequantize each weight block in registers and dot it with the input
 *    vector, one fused pass ("Что такое DMMV", habr ZINC article).
 *  - The dot is a packed int8x4 integer dot product accumulated into int32
 *    ("The reassuring result: ZINC's matmuls are __dp4a, not tensor cores",
 *    "Bringing ZINC to NVIDIA"; mapping table in "4. Kernel port strategy",
 *    "CUDA backend for ZINC").
 *  - Q4_0 values carry a -8 offset (Q4 snippet in "Что такое DMMV").
 *  - Q8_0/Q4_0 are 32-element GGML blocks, bit-for-bit the GGML layouts
 *    ("The reassuring result", "Bringing ZINC to NVIDIA").
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- fp16 ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN;
 * otherwise value = (1024 + fraction) * 2^(exponent - 25). */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest binary16, ties to even. The scaled
 * significand is formed exactly in binary64 and rounded with rint(), whose
 * default mode is round-to-nearest-even. */
uint16_t oracle_float_to_half_rne(float f)
{
    double v = (double)f;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return (uint16_t)(sign | 0x7e00);
    v = fabs(v);
    /* 65504 is the largest finite half; the midpoint to the next power of two
     * (65520) and everything above rounds to infinity under ties-to-even. */
    if (v >= 65520.0)
        return (uint16_t)(sign | 0x7c00);
    if (v < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24; a result of 1024 is the smallest
         * normal number and its bit pattern is exactly 0x0400 */
        double m = rint(v * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e2;
    frexp(v, &e2);          /* v = fr * 2^e2 with fr in [0.5, 1) */
    int expo = e2 - 1;      /* v in [2^expo, 2^(expo+1)) */
    double m = rint(v * ldexp(1.0, 10 - expo)); /* in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        expo += 1;
    }
    if (expo > 15)
        return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | ((expo + 15) << 10) | ((uint16_t)m - 1024));
}

/* ---------------------------------------------------------------- dp4a ---- */

int32_t oracle_dp4a(int32_t a, int32_t b, int32_t c)
{
    int64_t acc = c;
    for (int i = 0; i < 4; ++i) {
        int8_t ab = (int8_t)(uint8_t)(((uint32_t)a >> (8 * i)) & 0xff);
        int8_t bb = (int8_t)(uint8_t)(((uint32_t)b >> (8 * i)) & 0xff);
        acc += (int64_t)ab * (int64_t)bb;
    }
    return (int32_t)(uint32_t)(uint64_t)acc;
}

/* -------------------------------------------------------------- blocks ---- */

int oracle_block_bytes(int fmt)
{
    if (fmt == ORACLE_Q8_0)
        return 2 + 32;
    if (fmt == ORACLE_Q4_0)
        return 2 + 16;
    return 0;
}

static int quant_bytes(int fmt)
{
    return oracle_block_bytes(fmt) - 2;
}

int oracle_decode_block(int fmt, const uint8_t *blk, uint16_t *d_bits, int32_t q[32])
{
    *d_bits = (uint16_t)(blk[0] | (blk[1] << 8));
    if (fmt == ORACLE_Q8_0) {
        for (int i = 0; i < 32; ++i)
            q[i] = (int8_t)blk[2 + i];
        return 0;
    }
    if (fmt == ORACLE_Q4_0) {
        for (int j = 0; j < 16; ++j) {
            q[j] = (int32_t)(blk[2 + j] & 0x0f) - 8;
            q[j + 16] = (int32_t)(blk[2 + j] >> 4) - 8;
        }
        return 0;
    }
    return -1;
}

int oracle_dequantize(int fmt, const uint8_t *blocks, int64_t nblocks, double *out)
{
    int bb = oracle_block_bytes(fmt);
    if (bb == 0)
        return -1;
    for (int64_t i = 0; i < nblocks; ++i) {
        uint16_t dh;
        int32_t q[32];
        oracle_decode_block(fmt, blocks + i * bb, &dh, q);
        double d = oracle_half_to_double(dh);
        for (int j = 0; j < 32; ++j)
            out[32 * i + j] = d * (double)q[j];
    }
    return 0;
}

/* ------------------------------------------------------------ quantize ---- */

void oracle_quantize_q8_0(const float *x, int64_t k, uint8_t *xq)
{
    for (int64_t i = 0; i < k / 32; ++i) {
        const float *xb = x + 32 * i;
        uint8_t *blk = xq + 34 * i;
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax)
                amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        uint16_t dh = oracle_float_to_half_rne(d);
        blk[0] = (uint8_t)(dh & 0xff);
        blk[1] = (uint8_t)(dh >> 8);
        for (int j = 0; j < 32; ++j) {
            float v = xb[j] * id;
            float r = roundf(v);
            blk[2 + j] = (uint8_t)(int8_t)(int)r;
        }
    }
}

/* ---------------------------------------------------------------- DMMV ---- */

static int shape_ok(int fmt, int64_t rows, int64_t cols)
{
    return oracle_block_bytes(fmt) != 0 && rows >= 0 && cols > 0 && cols % 32 == 0;
}

/* s = sum_i qw_i * qx_i over one weight block and one Q8_0 activation block. */
static int64_t block_dot(int fmt, const uint8_t *wblk, const uint8_t *xblk,
                         uint16_t *dw, uint16_t *dx)
{
    int32_t qw[32], qx[32];
    oracle_decode_block(fmt, wblk, dw, qw);
    oracle_decode_block(ORACLE_Q8_0, xblk, dx, qx);
    int64_t s = 0;
    for (int i = 0; i < 32; ++i)
        s += (int64_t)qw[i] * (int64_t)qx[i];
    return s;
}

int oracle_block_sums(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                      const uint8_t *xq, int32_t *sums)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    int64_t nb = cols / 32;
    int bb = oracle_block_bytes(fmt);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            uint16_t dw, dx;
            int64_t s = block_dot(fmt, w + (r * nb + b) * bb, xq + b * 34, &dw, &dx);
            /* |s| <= 32*128*127 < 2^31: always representable as int32 */
            sums[r * nb + b] = (int32_t)s;
        }
    }
    return 0;
}

int oracle_dmmv(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                const uint8_t *xq, double *y, double *e)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    int64_t nb = cols / 32;
    int bb = oracle_block_bytes(fmt);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0, err = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            uint16_t dw, dx;
            int64_t s = block_dot(fmt, w + (r * nb + b) * bb, xq + b * 34, &dw, &dx);
            double t = oracle_half_to_double(dw) * oracle_half_to_double(dx) * (double)s;
            acc += t;
            err += fabs(t);
        }
        y[r] = acc;
        if (e)
            e[r] = err;
    }
    return 0;
}

/* The same product with the activation taken as fp32 values, not quantized:
 * each weight block is dequantized in registers and multiplied by the fp32
 * input vector (the ZINC_RT Q8_0 slice takes an f32 input vector: "The first
 * ZINC_RT model slices that actually count", the kernel ABI; the Vulkan DMMV
 * multiplies dequantized weights by an fp32 x staged in shared memory: habr
 * article, "Что такое DMMV" and "Трюк с shared memory"). In fp64:
 * y[r] = sum_b d_w * sum_i v_i * x_i, v_i the block's signed integer values. */
int oracle_dmmv_xf32(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                     const float *x, double *y, double *e)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    int64_t nb = cols / 32;
    int bb = oracle_block_bytes(fmt);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0, err = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            uint16_t dh;
            int32_t v[32];
            oracle_decode_block(fmt, w + (r * nb + b) * bb, &dh, v);
            double d = oracle_half_to_double(dh);
            double t = 0.0, ta = 0.0;
            for (int i = 0; i < 32; ++i) {
                double p = (double)v[i] * (double)x[b * 32 + i];
                t += p;
                ta += fabs(p);
            }
            acc += d * t;
            err += fabs(d) * ta;
        }
        y[r] = acc;
        if (e)
            e[r] = err;
    }
    return 0;
}

int oracle_dmmv_batched(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                        const uint8_t *xq, int batch, double *y, double *e)
{
    if (!shape_ok(fmt, rows, cols) || batch < 0)
        return -1;
    int64_t nb = cols / 32;
    for (int v = 0; v < batch; ++v) {
        int rc = oracle_dmmv(fmt, w, rows, cols, xq + (int64_t)v * nb * 34,
                             y + (int64_t)v * rows, e ? e + (int64_t)v * rows : NULL);
        if (rc)
            return rc;
    }
    return 0;
}

int oracle_expert_gather(int fmt, const uint8_t *w_stack, int64_t expert_stride_bytes,
                         int64_t rows, int64_t cols, const int32_t *idx, int n,
                         int n_experts, const uint8_t *xq, int64_t xq_stride_bytes,
                         double *y, double *e, int32_t *status)
{
    if (!shape_ok(fmt, rows, cols) || n < 0)
        return -1;
    for (int k = 0; k < n; ++k) {
        double *yk = y + (int64_t)k * rows;
        double *ek = e ? e + (int64_t)k * rows : NULL;
        if (idx[k] < 0 || idx[k] >= n_experts) {
            for (int64_t r = 0; r < rows; ++r) {
                yk[r] = NAN;
                if (ek)
                    ek[r] = NAN;
            }
            if (status)
                *status = 1;
            continue;
        }
        const uint8_t *wk = w_stack + (int64_t)idx[k] * expert_stride_bytes;
        const uint8_t *xk = xq + (int64_t)k * xq_stride_bytes;
        oracle_dmmv(fmt, wk, rows, cols, xk, yk, ek);
    }
    return 0;
}

/* ------------------------------------------------------------ epilogues ---- */

/* The shared expert's output is scaled by the sigmoid of its gate and added to
 * the MoE output ("sigmoid_scale_acc", M1 MoE chain in "CUDA backend for ZINC",
 * "5. The target model & milestone ordering"); with no gate the DMMV result is
 * simply accumulated (the templated DMMV's "accumulate mode", same section). */
int oracle_dmmv_acc(int fmt, const uint8_t *w, int64_t rows, int64_t cols, const uint8_t *xq,
                    const double *gate, double *y, double *e)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    double s = gate ? 1.0 / (1.0 + exp(-*gate)) : 1.0;
    double *d = (double *)malloc((size_t)(rows > 0 ? rows : 1) * 2 * sizeof(double));
    if (!d)
        return -1;
    double *de = d + (rows > 0 ? rows : 1);
    oracle_dmmv(fmt, w, rows, cols, xq, d, de);
    for (int64_t r = 0; r < rows; ++r) {
        y[r] += s * d[r];
        if (e)
            e[r] = s * de[r];
    }
    free(d);
    return 0;
}

/* The MoE expert FFN combines its gate and up projections with swiglu before the
 * down projection (M1 MoE chain "dmmv_q4k_moe gate/up + swiglu + dmmv_q5k_moe
 * down" and the fused "dmmv_*_fused_gate_up*" of M3: "CUDA backend for ZINC",
 * "5. The target model & milestone ordering"). The pages do not print the
 * formula; this is the standard SwiGLU: silu(gate) times up. */
void oracle_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* -------------------------------------------------------------- argmax ---- */

/* Greedy token pick over logits: the first index holding the maximum value
 * (argmax after the LM head: "Bringing ZINC to NVIDIA", section "The roadmap:
 * from 70 to a coherent token", the M1 forward order ending in argmax). */
int64_t oracle_argmax(const double *y, int64_t n, double *max_out)
{
    if (n <= 0)
        return -1;
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (y[i] > y[best])
            best = i;
    if (max_out)
        *max_out = y[best];
    return best;
}

/* -------------------------------------------------------------- repack ---- */

int oracle_repack(int fmt, const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    int64_t nb = cols / 32;
    int bb = oracle_block_bytes(fmt), qb = quant_bytes(fmt);
    uint8_t *scales = dst + rows * nb * qb;
    for (int64_t i = 0; i < rows * nb; ++i) {
        const uint8_t *blk = src + i * bb;
        scales[2 * i] = blk[0];
        scales[2 * i + 1] = blk[1];
        memcpy(dst + i * qb, blk + 2, (size_t)qb);
    }
    return 0;
}

int oracle_unpack(int fmt, const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst)
{
    if (!shape_ok(fmt, rows, cols))
        return -1;
    int64_t nb = cols / 32;
    int bb = oracle_block_bytes(fmt), qb = quant_bytes(fmt);
    const uint8_t *scales = src + rows * nb * qb;
    for (int64_t i = 0; i < rows * nb; ++i) {
        uint8_t *blk = dst + i * bb;
        blk[0] = scales[2 * i];
        blk[1] = scales[2 * i + 1];
        memcpy(blk + 2, src + i * qb, (size_t)qb);
    }
    return 0;
}
