/*
 * oracle.h -- plain, slow, CPU reference (the "oracle") for the GGUF Q8_0 / Q4_0
 * decode matrix-vector product y = W.x.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
 * call this code: only the test suite, the smoke check of the package entry
 * module and the CPU-baseline leg of the benchmark use it. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes (sources are the web pages this project restates):
 *  - "Bringing ZINC to NVIDIA: a CUDA backend" (zolotukhin.ai, 2026-06-06),
 *    section "The reassuring result: ZINC's matmuls are __dp4a, not tensor
 *    cores": quantized matvecs are packed int8x4 dot products accumulated into
 *    int32; GGML block layouts (Q8_0 = 32-element blocks) are bit-for-bit the
 *    GGML ones.
 *  - "CUDA backend for ZINC -- design & implementation plan", section
 *    "4. Kernel port strategy": the int8 dot maps to __dp4a; block layouts are
 *    identical to GGML's.
 *  - "Как мы запустили 35B LLM ... внутри ZINC inference engine" (habr), section
 *    "Что такое DMMV": read quantized weights, dequantize in registers, multiply
 *    by the input vector, write the result; the Q4 snippet there subtracts 8
 *    from each 4-bit value.
 *  - "The first ZINC_RT model slices that actually count", table in "What
 *    changed": Q4_0 and Q8_0 row-range DMMV slices.
 * Readings where the pages are silent (GGUF byte order of a block, nibble
 * order of Q4_0, rounding of the activation quantizer) follow the GGUF
 * standard and are listed in the design notes of the repository.
 *
 * Block formats (little-endian):
 *   Q8_0: bytes 0-1 fp16 scale d, bytes 2-33 int8 q[0..31];  value_i = d*q_i
 *   Q4_0: bytes 0-1 fp16 scale d, bytes 2-17 qs[0..15];
 *         q_j = qs[j] & 0xF, q_{j+16} = qs[j] >> 4 (j < 16);    value_i = d*(q_i-8)
 *
 * Repacked layout of a [rows x cols] matrix (nb = cols/32 blocks per row,
 * QB = 32 quant bytes for Q8_0, 16 for Q4_0):
 *   bytes [0, rows*nb*QB):            quant bytes of block (r,b) at (r*nb+b)*QB
 *   bytes [rows*nb*QB, rows*nb*(QB+2)): fp16 scale of block (r,b) at +(r*nb+b)*2
 */
#ifndef ZDMMV_ORACLE_H
#define ZDMMV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_Q4_0 = 2, ORACLE_Q8_0 = 8 };
enum { ORACLE_LAYOUT_GGUF = 0, ORACLE_LAYOUT_REPACKED = 1 };

/* IEEE-754 binary16 <-> binary64 / binary32, written from the format's definition. */
double   oracle_half_to_double(uint16_t h);
uint16_t oracle_float_to_half_rne(float f);

/* Packed int8x4 dot with int32 accumulate: c + sum_i a.byte_i * b.byte_i
 * (bytes as signed int8), the operation __dp4a performs. Wraps modulo 2^32. */
int32_t oracle_dp4a(int32_t a, int32_t b, int32_t c);

/* Bytes per block of a format (34 or 18); 0 for an unknown format. */
int oracle_block_bytes(int fmt);

/* Quantize k fp32 values (k % 32 == 0) into k/32 Q8_0 blocks:
 *   amax = max|x_i| (fp32); d = amax/127 (fp32); id = d ? 1/d : 0 (fp32);
 *   q_i = roundf(x_i*id) (fp32 product, ties away from zero); store fp16(d) (RNE). */
void oracle_quantize_q8_0(const float *x, int64_t k, uint8_t *xq);

/* Decode one block into its fp16 scale bits and 32 signed integer values
 * (Q4_0 values already have the -8 offset applied). Returns 0, or -1 for an
 * unknown format. */
int oracle_decode_block(int fmt, const uint8_t *blk, uint16_t *d_bits, int32_t q[32]);

/* Dequantize nblocks blocks into 32*nblocks doubles: d*q_i (Q8_0) or d*(q_i-8) (Q4_0). */
int oracle_dequantize(int fmt, const uint8_t *blocks, int64_t nblocks, double *out);

/* Integer per-block dot products s[r*nb+b] = sum_i qw_i*qx_i of weight block
 * (r,b) (GGUF layout) against activation block b (Q8_0). */
int oracle_block_sums(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                      const uint8_t *xq, int32_t *sums);

/* y[r] = sum_b fp16(d_w)*fp16(d_x)*s_b, in fp64, in block order; e[r] =
 * sum_b |fp16(d_w)*fp16(d_x)*s_b| (the per-row error scale). w is GGUF layout. */
int oracle_dmmv(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                const uint8_t *xq, double *y, double *e);

/* y[r] = sum_b d_w * sum_i v_i * x_i with the activation x taken as fp32 values
 * (no quantization); v_i are the block's signed values (Q4_0: q - 8). e[r] =
 * sum_b sum_i |d_w * v_i * x_i|. Computed in fp64. */
int oracle_dmmv_xf32(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                     const float *x, double *y, double *e);

/* The same for `batch` activation vectors stored [batch][cols/32] blocks;
 * y and e are [batch][rows]. */
int oracle_dmmv_batched(int fmt, const uint8_t *w, int64_t rows, int64_t cols,
                        const uint8_t *xq, int batch, double *y, double *e);

/* Expert gather: for k < n, W_k = w_stack + idx[k]*expert_stride_bytes and
 * x_k = xq + k*xq_stride_bytes (0 = one shared vector); y[k][rows] = W_k . x_k.
 * An index outside [0, n_experts) gives NaN rows and sets *status = 1.
 * Returns 0 or -1 (unknown format / bad shape). */
int oracle_expert_gather(int fmt, const uint8_t *w_stack, int64_t expert_stride_bytes,
                         int64_t rows, int64_t cols, const int32_t *idx, int n,
                         int n_experts, const uint8_t *xq, int64_t xq_stride_bytes,
                         double *y, double *e, int32_t *status);

/* Accumulate epilogue: y[r] += s * (W.x)[r] with s = 1 when gate is NULL, else
 * s = sigmoid(*gate) = 1 / (1 + exp(-*gate)) (fp64). y is updated in place;
 * e[r] (nullable) receives s * sum_b |d_w d_x s_b|. */
int oracle_dmmv_acc(int fmt, const uint8_t *w, int64_t rows, int64_t cols, const uint8_t *xq,
                    const double *gate, double *y, double *e);

/* SwiGLU of the gate and up projections: h_i = silu(g_i) * u_i with
 * silu(g) = g / (1 + exp(-g)) (fp64). */
void oracle_swiglu(const double *g, const double *u, int64_t n, double *h);

/* Index of the largest of n values (the smallest such index on ties), or -1 for
 * n <= 0; the greedy pick over the LM-head logits. *max_out receives the value. */
int64_t oracle_argmax(const double *y, int64_t n, double *max_out);

/* GGUF array-of-blocks -> repacked (quant stream + scale array), and back. */
int oracle_repack(int fmt, const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst);
int oracle_unpack(int fmt, const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst);

#ifdef __cplusplus
}
#endif

#endif /* ZDMMV_ORACLE_H */
