/*
 * zdmmv.h -- C ABI of the GB300 (sm_103a) GGUF block-quantized decode DMMV
 * library (libzdmmv.so).
 *
 * The operation. A decode DMMV ("dequantize matrix x vector") computes
 * y = W.x for one decode token: it reads the quantized weights once,
 * dequantizes them in registers, multiplies by the input vector and writes the
 * result, with no intermediate dequantized buffer (habr article "Как мы
 * запустили 35B LLM ... внутри ZINC inference engine", section "Что такое DMMV";
 * decode is bound by memory bandwidth, section "Ядро: DMMV и борьба за
 * пропускную способность памяти"). The arithmetic is a packed int8x4 integer
 * dot product accumulated in int32 -- GL_EXT_integer_dot_product on Vulkan,
 * __dp4a in CUDA ("Bringing ZINC to NVIDIA: a CUDA backend", section "The
 * reassuring result: ZINC's matmuls are __dp4a, not tensor cores"; "CUDA
 * backend for ZINC -- design & implementation plan", section "4. Kernel port
 * strategy"). Per 32-element block b of row r:
 *     s_b  = sum_{i<32} qw_i * qx_i                      (int32, exact)
 *     y_r  = sum_b fp16(d_w[r,b]) * fp16(d_x[b]) * s_b    (fp32 accumulation)
 * where qw_i is the Q8_0 int8 value, or the Q4_0 4-bit value minus 8 (the -8
 * offset of the Q4 unpack in "Что такое DMMV"), and qx_i / d_x come from the
 * activation quantized to Q8_0 blocks by zdmmv_quantize_act_q8_0.
 *
 * Block formats (GGML/GGUF layouts, bit-for-bit; "The reassuring result",
 * "Bringing ZINC to NVIDIA"), little-endian:
 *     Q8_0 (34 B): fp16 d, int8 q[32];                  value = d*q
 *     Q4_0 (18 B): fp16 d, uint8 qs[16]; element j = qs[j] & 15,
 *                  element j+16 = qs[j] >> 4 (j < 16);   value = d*(q-8)
 * A [rows x cols] matrix in ZDMMV_LAYOUT_GGUF is rows*cols/32 blocks, row-major.
 * ZDMMV_LAYOUT_REPACKED (produced by zdmmv_repack) keeps the same bytes as a
 * quant stream (block (r,b) at (r*nb+b)*QB, QB = 32 or 16) followed by an fp16
 * scale array (block (r,b) at rows*nb*QB + (r*nb+b)*2), nb = cols/32.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev / w / xq / y are DEVICE pointers owned by the caller;
 *    the library never allocates, frees or retains them.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). Argument errors are returned synchronously before any
 *    launch; launch failures return ZDMMV_ERR_CUDA. No entry point
 *    synchronizes the device except zdmmv_device_status.
 *  - Weight matrices are treated as read-only model parameters: with
 *    programmatic dependent launch the DMMV kernels start streaming weight
 *    tiles before the preceding kernel in the stream has finished (activations,
 *    expert indices and outputs are touched only after it has, except the index
 *    list of the ready gathers, zdmmv_expert_gather_ready and
 *    zdmmv_expert_gather_f32 with idx_ready, under their stated requirement). A
 *    weight buffer
 *    must therefore be complete before the DMMV that reads it is enqueued
 *    behind a kernel still writing it; enqueue an event or synchronize in
 *    between if weights are produced on the device (zdmmv_repack's output may
 *    be used directly: its kernel never releases dependents early). Set the
 *    environment variable ZDMMV_PDL=0 to disable programmatic dependent launch.
 *  - Launch-shape tuning, read once per process from the environment (all
 *    optional; results are the same bits whatever they are set to unless stated):
 *      ZDMMV_STAGE_KB           target KiB per pipeline stage (4..64, default 20)
 *      ZDMMV_CTAS_PER_SM        CTAs per SM of the single-vector kernel (1..8;
 *                               default 2 below 32 MB of weights per launch, else 4;
 *                               expert gathers that wait for their indices as many
 *                               as fit)
 *      ZDMMV_BATCH_KERNEL       batched kernel (see zdmmv_q8_0_batched for the
 *                               default choice): "vsplit" (the vector split, never
 *                               the tensor-core kernel), "mma" (the tensor-core
 *                               kernel wherever it takes the shape, 2..8 vectors,
 *                               else the vector split), "stream", or "slots" (one
 *                               single-vector slot per vector). Every choice keeps
 *                               the result within the stated tolerance; the fp32
 *                               reduction order of batch > 1 follows the kernel
 *                               (for "vsplit" and "slots" it is the single-vector
 *                               order)
 *      ZDMMV_BATCH_SLOTS=1      the same as ZDMMV_BATCH_KERNEL=slots
 *      ZDMMV_VSPLIT_V=1         one vector per warp in the vector-split kernel;
 *                               batches of more than 4 vectors that the
 *                               tensor-core kernel does not take then take the
 *                               "stream" kernel (its fp32 reduction order)
 *      ZDMMV_BATCH_CTAS_PER_SM  CTAs per SM of the batched kernels (1..4)
 *      ZDMMV_FFN_STAGES=3       three pipeline stages in zdmmv_expert_ffn (default 2)
 *      ZDMMV_FFN_CTAS_PER_SM    CTAs per SM of zdmmv_expert_ffn (1..8, default as
 *                               many as fit)
 *      ZDMMV_FFN_GU_PERCENT     share of zdmmv_expert_ffn's CTAs on gate/up rows
 *                               (20..80, default 60; the rest on down rows)
 *  - There is no CPU fallback: every result is computed by the CUDA kernels.
 *  - Inputs must be finite (a NaN or infinite activation gives unspecified
 *    codes).
 */
#ifndef ZDMMV_H
#define ZDMMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *); declared here so the
 * header needs no CUDA include. */
typedef struct CUstream_st *zdmmv_stream_t;

typedef enum {
    ZDMMV_OK = 0,
    ZDMMV_ERR_NULL = 1,    /* a required pointer is NULL */
    ZDMMV_ERR_SHAPE = 2,   /* cols <= 0, cols % 32 != 0, rows < 0, k % 32 != 0,
                              batch outside 1..8, n < 0, bad strides */
    ZDMMV_ERR_ALIGN = 3,   /* w, xq or a stride not 16-byte aligned; x, y not 4-byte aligned */
    ZDMMV_ERR_LAYOUT = 4,  /* unknown layout */
    ZDMMV_ERR_FORMAT = 5,  /* unknown block format */
    ZDMMV_ERR_SIZE = 6,    /* destination or workspace too small */
    ZDMMV_ERR_CUDA = 7,    /* a CUDA runtime call or a kernel launch failed */
    ZDMMV_ERR_DEVICE = 8   /* a kernel reported a fault (see zdmmv_device_status) */
} zdmmv_status;

typedef enum { ZDMMV_Q4_0 = 2, ZDMMV_Q8_0 = 8 } zdmmv_fmt;     /* GGML type ids */
typedef enum { ZDMMV_LAYOUT_GGUF = 0, ZDMMV_LAYOUT_REPACKED = 1 } zdmmv_layout;

#define ZDMMV_QK 32         /* elements per block */
#define ZDMMV_MAX_BATCH 8   /* activation vectors per batched call */

/* Device fault bits reported by zdmmv_device_status. */
#define ZDMMV_FAULT_WAIT_TIMEOUT 1u  /* a bounded wait on a copy or a pipeline stage gave up */
#define ZDMMV_FAULT_SMEM_ALIGN   2u  /* a kernel found its shared-memory stages off the
                                        alignment its tensor copies need and computed nothing */

/* Human-readable name of a status code (static string). */
const char *zdmmv_status_str(zdmmv_status st);

/* Library version string (static). */
const char *zdmmv_version(void);

/* Bytes of one block of `fmt` (34 or 18), 0 for an unknown format. */
size_t zdmmv_block_bytes(zdmmv_fmt fmt);

/* Quantize k fp32 activations to k/32 Q8_0 blocks (34 B each), per block:
 *   amax = max|x_i|; d = amax/127 (fp32, IEEE division); id = d ? 1/d : 0;
 *   q_i = round(x_i*id) (fp32 product, ties away from zero); store fp16(d)
 *   (round to nearest even) then q[32].
 * This is the activation quantizer that feeds the int8 dot (the "quantize"
 * shaders in "Bringing ZINC to NVIDIA", section "Porting the kernels"; the
 * rounding reading is the GGUF reference quantizer's, since the pages do not
 * print it). A batch of vectors stored back to back is one call with k =
 * batch*cols.
 *   x   device, k floats, 4-byte aligned;   xq device, k/32*34 bytes.
 *   k   multiple of 32; k == 0 is a no-op.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_CUDA. */
zdmmv_status zdmmv_quantize_act_q8_0(const float *x, int64_t k, void *xq,
                                     zdmmv_stream_t stream);

/* y = W.x for one activation vector (Q8_0 or Q4_0 weights).
 *   w      device, the matrix in `layout`, 16-byte aligned.
 *   rows   >= 0 (0 is a no-op);  cols > 0, multiple of 32.
 *   xq     device, cols/32 Q8_0 activation blocks, 16-byte aligned.
 *   y      device, rows floats (fp32), 4-byte aligned.
 * Matrices whose rows are 16-byte multiples (cols % 256 == 0) and cols <= 8192
 * take the TMA-pipelined kernel; other shapes take a plain kernel with the
 * same arithmetic. Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_CUDA. */
zdmmv_status zdmmv_q8_0(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                        const void *xq, float *y, zdmmv_stream_t stream);
zdmmv_status zdmmv_q4_0(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                        const void *xq, float *y, zdmmv_stream_t stream);

/* The same weight matrix against `batch` (1..8) activation vectors in one call:
 * xq is [batch][cols/32] Q8_0 blocks, y is [batch][rows] fp32. Each weight tile
 * is streamed from HBM once and dotted against every vector (concurrency
 * headroom of decode slots: habr article, section "RDNA4: что мы узнали о
 * железе"). Default kernels:
 *  - batch 5..8, GGUF layout, widths that are multiples of 256 from 1280 to
 *    4096 columns, and at least 32 rows per SM of the device (4864 rows on a
 *    152-SM GB300): the fp16 tensor-core kernel. Each block's integer dot
 *    product is exact (the pages' int32 block sum) and its scales are applied in
 *    fp32, but the blocks of a row are summed in another order than the
 *    single-vector kernel's: deterministic, within the stated tolerance, not
 *    bit for bit zdmmv_q8_0 on each vector;
 *  - other widths that are multiples of 256 up to 4096 columns (up to 8192 with
 *    batch <= 4): the consumer warps split the vectors and every vector's result
 *    is the single-vector computation, bit for bit: y[v] equals zdmmv_q8_0 /
 *    zdmmv_q4_0 on vector v;
 *  - widths of 8192 columns with batch > 4 stream the tile through a kernel
 *    whose fp32 reduction order differs (deterministic, within the stated
 *    tolerance); other widths run the single-vector computation once per
 *    vector.
 * batch == 1 is zdmmv_q8_0 / zdmmv_q4_0. The environment variable
 * ZDMMV_BATCH_KERNEL (above) selects other kernels.
 * Errors: as zdmmv_q8_0, plus ERR_SHAPE for batch outside 1..8. */
zdmmv_status zdmmv_q8_0_batched(const void *w, zdmmv_layout layout, int64_t rows,
                                int64_t cols, const void *xq, int batch, float *y,
                                zdmmv_stream_t stream);
zdmmv_status zdmmv_q4_0_batched(const void *w, zdmmv_layout layout, int64_t rows,
                                int64_t cols, const void *xq, int batch, float *y,
                                zdmmv_stream_t stream);

/* Fused decode step: the same result as zdmmv_quantize_act_q8_0 followed by
 * zdmmv_q{8,4}_0_batched (zdmmv_q{8,4}_0 for batch 1), bit for bit, in ONE
 * launch. Each CTA quantizes the fp32 activation to Q8_0 blocks in shared memory
 * itself, so a chain of decode layers pays one kernel per layer instead of two
 * (per-token launch chains: "RTX 5090: Batched Prefill & CUDA Graphs in ZINC",
 * "CUDA graphs -- the structural answer to launch latency"). So where the
 * batched call is the single-vector computation per vector, so is this one;
 * where it takes the tensor-core kernel (5..8 vectors, see
 * zdmmv_q8_0_batched), this one does too.
 *   fmt    ZDMMV_Q8_0 or ZDMMV_Q4_0 weights; w, layout, rows, cols as zdmmv_q8_0.
 *   x      device fp32 [batch][cols], 16-byte aligned; batch 1..8.
 *   y      device fp32 [batch][rows].
 * Batches of 2..8 on the batched kernels' shapes stream the weights once (every
 * CTA quantizes the whole batch); other batches run one fused launch with a
 * slot per vector. For batches the two calls (zdmmv_quantize_act_q8_0, then
 * zdmmv_q{8,4}_0_batched) are faster: the quantization is done once instead of
 * in every CTA.
 * Shapes off the pipelined path (cols % 256 != 0 or cols > 8192) need
 * batch*cols/32*34 <= 200 KiB of shared memory, else ERR_SHAPE.
 * Errors: as zdmmv_q8_0_batched, plus ERR_FORMAT. */
zdmmv_status zdmmv_dmmv_f32(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows,
                            int64_t cols, const float *x, int batch, float *y,
                            zdmmv_stream_t stream);

/* The product with the activation taken as fp32 values, NOT quantized:
 * y[v][r] = sum_b d_w * sum_i v_i * x[v][32b + i], v_i the weight block's signed
 * values (Q4_0: q - 8). Each weight block is dequantized in registers and
 * multiplied by the fp32 x staged in shared memory, the form of the ZINC_RT
 * Q8_0 slice (f32 input vector: "The first ZINC_RT model slices that actually
 * count", kernel ABI) and of the Vulkan DMMV's shared-memory x (habr article,
 * "Что такое DMMV", "Трюк с shared memory"). It reads 4 bytes per activation
 * element instead of 34/32 and spends an fp32 fma per weight instead of a dp4a
 * per four: an accuracy reference for the quantized-activation path.
 *   fmt, w, layout, rows, cols   as zdmmv_dmmv_f32 (any multiple of 32 columns;
 *                                widths off the pipelined path run a plain kernel).
 *   x      device fp32 [batch][cols], 16-byte aligned; batch 1..8.
 *   y      device fp32 [batch][rows].
 * Results are fp32 sums within 1e-5 * sum_b sum_i |d_w v_i x_i| + 1e-6 of the
 * exact product, deterministic from call to call.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_FORMAT, ERR_CUDA. */
zdmmv_status zdmmv_dmmv_xf32(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows,
                             int64_t cols, const float *x, int batch, float *y,
                             zdmmv_stream_t stream);

/* Accumulate epilogue: y[r] = y[r] + s * (W.x)[r], one fused fma per row, with
 * s = 1 when gate is NULL (the templated DMMV's "accumulate mode") or
 * s = sigmoid(*gate) = 1/(1 + exp(-*gate)) for a device fp32 gate scalar (the
 * shared expert's "sigmoid_scale_acc"; both in "CUDA backend for ZINC",
 * "5. The target model & milestone ordering", M1). The gate and y may be
 * written by the preceding kernel in the stream.
 *   fmt, w, layout, rows, cols, xq   as zdmmv_q8_0 (any width that is a
 *                                    multiple of 32).
 *   gate   nullable device float[1].
 *   y      device fp32 [rows], read and written.
 * Errors: as zdmmv_q8_0, plus ERR_FORMAT. */
zdmmv_status zdmmv_dmmv_acc(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows,
                            int64_t cols, const void *xq, const float *gate, float *y,
                            zdmmv_stream_t stream);

/* Gate and up projections of the selected experts with the SwiGLU epilogue,
 * in ONE launch: h[k][r] = silu(G_{idx[k]}.x_k)[r] * (U_{idx[k]}.x_k)[r] with
 * silu(g) = g / (1 + exp(-g)). The MoE step runs the gate/up DMMV and then
 * swiglu ("CUDA backend for ZINC", "5. The target model & milestone ordering",
 * M1), the plan fuses gate and up into one launch (M3,
 * "dmmv_*_fused_gate_up*"), and the habr article counts the separate SiLU and
 * multiply passes as avoidable traffic ("Fused операции"). Each CTA streams the
 * same row tile of both matrices into one pipeline stage, so the two dot
 * products of a row are formed side by side and only h is written.
 *   fmt, layout, rows, cols  as zdmmv_q8_0; cols must be a multiple of 256 and
 *                            at most 8192 (else ERR_SHAPE).
 *   w_gate, w_up   device stacks of the same shape: expert e's matrices start at
 *                  w_gate + e*expert_stride_bytes and w_up + e*expert_stride_bytes
 *                  (16-byte multiple). With idx == NULL they are one gate and one
 *                  up matrix (a dense FFN), n must be 1 and expert_stride_bytes
 *                  and n_experts are ignored.
 *   idx            nullable DEVICE int32[n], read by the kernel.
 *   n              number of slots (0..65535; 0 is a no-op).
 *   xq, xq_stride_bytes, status_dev   as zdmmv_expert_gather.
 *   h              device fp32 [n][rows].
 * The gate and up dot products are the fp32 values zdmmv_expert_gather2 writes,
 * bit for bit; h is silu(g)*u of those in fp32 (an IEEE divide by 1 + expf(-g)
 * and one multiply), within a few ulp of silu in exact arithmetic.
 * Errors: as zdmmv_expert_gather. */
zdmmv_status zdmmv_expert_swiglu(zdmmv_fmt fmt, const void *w_gate, const void *w_up,
                                 int64_t expert_stride_bytes, zdmmv_layout layout,
                                 int64_t rows, int64_t cols, const int32_t *idx, int n,
                                 int n_experts, const void *xq, int64_t xq_stride_bytes,
                                 float *h, int32_t *status_dev, zdmmv_stream_t stream);

/* The selected experts' whole FFN in ONE launch: for k < n, with e = idx[k],
 *   h_k = silu(G_e . x) * (U_e . x)            (gate/up DMMVs, SwiGLU epilogue)
 *   y_k = D_e . q8_0(h_k)                       (down DMMV of the quantized h_k)
 * the MoE step's gate/up DMMV, swiglu and down DMMV ("CUDA backend for ZINC",
 * "5. The target model & milestone ordering", M1) as one dispatch for all
 * experts (habr article, "Gap analysis"; "RTX 5090: Batched Prefill & CUDA
 * Graphs in ZINC", "What's next"). One grid holds gate/up CTAs and down CTAs;
 * the down CTAs stream their weights while the gate/up CTAs run, then wait
 * (bounded) on a per-expert counter in the workspace before reading h_k.
 *   fmt_gate_up  format of the gate and up stacks (Q4_0 or Q8_0), GGUF layout;
 *                expert e's [ffn x hidden] matrices at w_gate / w_up +
 *                e*gate_up_stride_bytes.
 *   fmt_down     format of the down stack, GGUF layout; expert e's [hidden x ffn]
 *                matrix at w_down + e*down_stride_bytes. Strides are 16-byte
 *                multiples (>= the matrix size when n_experts > 1).
 *   hidden       a multiple of 256, at most 4096; ffn a multiple of 256, at most
 *                2048 (else ERR_SHAPE). n == 0 is a no-op.
 *   idx, n, n_experts, status_dev   as zdmmv_expert_gather; n <= 4096 and at
 *                most half the CTAs that fit on the device at once (every CTA of
 *                the grid must be resident: 380 on a 152-SM GB300 at 5 CTAs per SM),
 *                else ERR_SHAPE; a bad
 *                index gives NaN rows of h_k and y_k.
 *   xq           device Q8_0 blocks of the hidden activation, shared by all slots.
 *   y            device fp32 [n][hidden].
 *   workspace    device, 256-byte aligned, >= zdmmv_expert_ffn_workspace_bytes(n,
 *                ffn) bytes, ZERO-FILLED before its first use; every call leaves
 *                its counters zero again. Bytes [0, 4*n*ffn) hold h after the
 *                call. One workspace per call in flight. After a call that
 *                reported ZDMMV_FAULT_WAIT_TIMEOUT, zero it again.
 * h_k is the zdmmv_expert_swiglu value and y_k the zdmmv_expert_gather value on
 * zdmmv_quantize_act_q8_0(h_k), bit for bit. The same results come from two
 * launches, zdmmv_expert_swiglu and then zdmmv_expert_gather_f32 of h with
 * idx_ready set, which measured faster on a GB300 (8 routed + 1 shared expert,
 * hidden 2048, ffn 512: 7.9 against 9.0 us per token and layer): the down
 * gather's weights stream during the SwiGLU launch, where here the down CTAs
 * wait on per-expert counters.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_FORMAT, ERR_SIZE, ERR_CUDA. */
size_t zdmmv_expert_ffn_workspace_bytes(int n, int64_t ffn);
zdmmv_status zdmmv_expert_ffn(zdmmv_fmt fmt_gate_up, const void *w_gate, const void *w_up,
                              int64_t gate_up_stride_bytes, zdmmv_fmt fmt_down, const void *w_down,
                              int64_t down_stride_bytes, int64_t hidden, int64_t ffn,
                              const int32_t *idx, int n, int n_experts, const void *xq, float *y,
                              void *workspace, size_t workspace_bytes, int32_t *status_dev,
                              zdmmv_stream_t stream);

/* LM-head DMMV with a fused argmax epilogue: the greedy pick over the logits
 * W.x without writing them (the M1 decode chain ends "LM head -> argmax":
 * "Bringing ZINC to NVIDIA", section "The roadmap: from 70 to a coherent
 * token"; the logits tail is part of the per-token time in the habr article,
 * "Разбивка по времени"). Each CTA keeps the largest logit of its rows and the
 * first row holding it, writes one 8-byte partial into `workspace`, and a
 * one-CTA pass reduces the partials. The logits are the same fp32 values
 * zdmmv_q{8,4}_0 would write (same kernel arithmetic), so the result is the
 * first index of their maximum.
 *   w, layout, rows (1 .. 2^31-1), cols, xq   as zdmmv_q8_0; cols must be a
 *            multiple of 256 and at most 8192 (else ERR_SHAPE).
 *   argmax_out  device int32[1]: the row index.
 *   max_out     nullable device float[1]: the logit at that row.
 *   workspace   caller-owned device scratch, 16-byte aligned, of at least
 *               ZDMMV_ARGMAX_WORKSPACE_BYTES; overwritten by each call, so two
 *               calls in flight at once need two workspaces.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_FORMAT, ERR_SIZE, ERR_CUDA. */
#define ZDMMV_ARGMAX_WORKSPACE_BYTES 16384
zdmmv_status zdmmv_dmmv_argmax(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows,
                               int64_t cols, const void *xq, int32_t *argmax_out, float *max_out,
                               void *workspace, size_t workspace_bytes, zdmmv_stream_t stream);

/* The same greedy pick as zdmmv_dmmv_argmax for callers that cannot allocate
 * device memory: an engine that plans all device memory when it loads a model
 * and treats any later allocation as a bug, a plugin whose host program owns
 * every device allocation, or a decode loop that must not call cudaMalloc
 * (which may synchronize the device). No workspace argument; the per-CTA
 * partials go to a fixed 16 KiB array inside the library's device image
 * (2048 slots), which every GPU that loads the library holds until the process
 * exits. The pages have no counterpart of this entry point; it is an addition
 * of this library.
 *   Arguments as zdmmv_dmmv_argmax without workspace / workspace_bytes; rows
 *   1 .. 2^31-1 (a launch never needs more than the 2048 slots), cols a
 *   multiple of 256 and at most 8192; anything else is ERR_SHAPE.
 *   Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Every call shares the array and leaves the last call's partials in it
 *   (nothing needs to start at zero: each call writes every slot it reads).
 *   Calls that overlap on the GPU (other streams or threads) race on the array
 *   and may return wrong results; serialize them.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_FORMAT, ERR_CUDA. */
zdmmv_status zdmmv_dmmv_argmax_noalloc(zdmmv_fmt fmt, const void *w, zdmmv_layout layout,
                                       int64_t rows, int64_t cols, const void *xq,
                                       int32_t *argmax_out, float *max_out,
                                       zdmmv_stream_t stream);

/* MoE expert gather: n matrices picked by index from a stack of n_experts
 * equally shaped matrices, all in ONE launch (routed experts are selected per
 * token by the router: "CUDA backend for ZINC", M1 list "dmmv_q4k_moe";
 * batching the experts into one dispatch: habr article, sections "Gap
 * analysis" and "Что дальше"; a GPU-side gather that drops the router
 * round-trip: "RTX 5090: Batched Prefill & CUDA Graphs in ZINC", "What's next").
 *   w_stack             device; expert e starts at w_stack + e*expert_stride_bytes
 *                       (16-byte multiple), each a [rows x cols] matrix in `layout`.
 *   idx                 DEVICE int32[n], read by the kernel (no host round-trip).
 *   n                   number of selected experts (0..32767; 0 is a no-op).
 *   n_experts           valid indices are 0 .. n_experts-1.
 *   xq                  device Q8_0 blocks; slot k reads xq + k*xq_stride_bytes
 *                       (xq_stride_bytes = 0: one activation shared by all slots;
 *                       otherwise a 16-byte multiple >= cols/32*34).
 *   y                   device fp32 [n][rows].
 *   status_dev          nullable device int32; an index outside [0, n_experts)
 *                       fills that slot's rows with NaN and stores 1 here. The
 *                       kernel never reads out of range for a bad index.
 * Slot k's result equals zdmmv_q{8,4}_0 on matrix idx[k], bit for bit.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_FORMAT, ERR_CUDA. */
zdmmv_status zdmmv_expert_gather(zdmmv_fmt fmt, const void *w_stack,
                                 int64_t expert_stride_bytes, zdmmv_layout layout,
                                 int64_t rows, int64_t cols, const int32_t *idx, int n,
                                 int n_experts, const void *xq, int64_t xq_stride_bytes,
                                 float *y, int32_t *status_dev, zdmmv_stream_t stream);

/* zdmmv_expert_gather for a selection that an earlier expert call has already
 * read: the down projections after the gate/up launch of the same experts, or
 * the up projections after the gates' gather (the MoE step's gate/up DMMV, then
 * the down DMMV of the same routed experts: "CUDA backend for ZINC", "5. The
 * target model & milestone ordering", M1). zdmmv_expert_gather must wait for
 * the preceding kernel before it reads idx, so its weights cannot stream until
 * then; this call reads idx as soon as its kernel starts and streams its first
 * weight tiles while the preceding kernel still runs. It waits for that kernel
 * before it reads xq or writes y, so xq (and y) may be written (read) by it.
 *   Arguments, results (bit for bit) and errors as zdmmv_expert_gather.
 *   Requirement on idx: an earlier call among zdmmv_expert_gather,
 *   zdmmv_expert_gather2, zdmmv_expert_swiglu and zdmmv_expert_gather_ready that
 *   this call is ordered after (the same stream, or an event) read the same
 *   device list, with its final contents, and nothing has written the list since.
 *   Those calls let later launches start only once their own index list is
 *   complete (after their dependency wait), so the list this call reads is
 *   complete too. Without that earlier call the kernel may read a list that the
 *   preceding kernel is still writing: use zdmmv_expert_gather. */
zdmmv_status zdmmv_expert_gather_ready(zdmmv_fmt fmt, const void *w_stack,
                                       int64_t expert_stride_bytes, zdmmv_layout layout,
                                       int64_t rows, int64_t cols, const int32_t *idx, int n,
                                       int n_experts, const void *xq, int64_t xq_stride_bytes,
                                       float *y, int32_t *status_dev, zdmmv_stream_t stream);

/* Expert gather over fp32 activations, quantized to Q8_0 inside the launch: the
 * MoE step's down DMMV of the SwiGLU output h without a separate quantizer
 * launch (M1's gate/up DMMV, swiglu, down DMMV: "CUDA backend for ZINC", "5. The
 * target model & milestone ordering"; fewer dispatches per token: habr article,
 * "Gap analysis"). Each CTA quantizes its slot's activation into shared memory
 * with the arithmetic of zdmmv_quantize_act_q8_0, so slot k's result equals
 * zdmmv_quantize_act_q8_0 of x_k followed by zdmmv_expert_gather, bit for bit.
 *   fmt, w_stack, expert_stride_bytes, layout, rows, idx, n, n_experts,
 *   status_dev   as zdmmv_expert_gather; cols a multiple of 256 and at most 8192
 *                (else ERR_SHAPE).
 *   x            device fp32, 16-byte aligned; slot k reads x + k*x_stride
 *                (x_stride in floats: 0 = one activation shared by all slots,
 *                else a multiple of 4 and >= cols). x may be written by the
 *                preceding kernel in the stream (e.g. zdmmv_expert_swiglu's h).
 *   y            device fp32 [n][rows].
 *   idx_ready    0: read idx after waiting for the preceding kernel, as
 *                zdmmv_expert_gather; nonzero: read it at once and stream weights
 *                early, under zdmmv_expert_gather_ready's requirement on idx.
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_FORMAT, ERR_CUDA. */
zdmmv_status zdmmv_expert_gather_f32(zdmmv_fmt fmt, const void *w_stack,
                                     int64_t expert_stride_bytes, zdmmv_layout layout,
                                     int64_t rows, int64_t cols, const int32_t *idx, int n,
                                     int n_experts, const float *x, int64_t x_stride, float *y,
                                     int32_t *status_dev, int idx_ready, zdmmv_stream_t stream);

/* Two expert stacks of the same shape and format against the same selected
 * experts and activations, in ONE launch: y_a[k] = A_{idx[k]} . x_k and
 * y_b[k] = B_{idx[k]} . x_k (the gate and up projections of the routed experts,
 * which the pages plan as one fused launch: "CUDA backend for ZINC", M3
 * "dmmv_*_fused_gate_up*"; same-input matvec pairs fused: "RTX 5090: Batched
 * Prefill & CUDA Graphs in ZINC", "Gemma fusion"). Arguments as
 * zdmmv_expert_gather, with the two stacks sharing expert_stride_bytes; y_a and
 * y_b are [n][rows]. Each output equals zdmmv_expert_gather on its own stack,
 * bit for bit. Errors: as zdmmv_expert_gather. */
zdmmv_status zdmmv_expert_gather2(zdmmv_fmt fmt, const void *w_stack_a, const void *w_stack_b,
                                  int64_t expert_stride_bytes, zdmmv_layout layout, int64_t rows,
                                  int64_t cols, const int32_t *idx, int n, int n_experts,
                                  const void *xq, int64_t xq_stride_bytes, float *y_a, float *y_b,
                                  int32_t *status_dev, zdmmv_stream_t stream);

/* Bytes of the repacked form of a [rows x cols] matrix (equal to the GGUF size);
 * 0 for an unknown format or a bad shape. */
size_t zdmmv_repacked_bytes(zdmmv_fmt fmt, int64_t rows, int64_t cols);

/* One-time repack of a GGUF-layout matrix into ZDMMV_LAYOUT_REPACKED (a
 * 16-byte aligned quant stream plus a separate fp16 scale array; the pages'
 * shaders read 128-bit vec4/uvec4 words: "CUDA backend for ZINC", "4. Kernel
 * port strategy"). Pure byte permutation, bit-exact.
 *   src, dst   device, 16-byte aligned, must not overlap; dst_bytes >=
 *              zdmmv_repacked_bytes(fmt, rows, cols).
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_FORMAT, ERR_SIZE, ERR_CUDA. */
zdmmv_status zdmmv_repack(zdmmv_fmt fmt, const void *src, int64_t rows, int64_t cols,
                          void *dst, size_t dst_bytes, zdmmv_stream_t stream);

/* One decode step with HOST activations and outputs: x_host ([batch][cols]
 * fp32) in, y_host ([batch][rows] fp32) out, quantized and multiplied on the
 * resident weights, all ordered on `stream`. When each buffer lies in one
 * page-locked allocation mapped into the device's address space (cudaHostAlloc,
 * torch pin_memory), the kernels use the host memory in place: the quantizer
 * reads x_host and the DMMV stores y_host (over the chip-to-chip link on a
 * Grace system; no copy calls). Otherwise x is copied to the workspace, the
 * fused quantize + DMMV (as zdmmv_dmmv_f32) runs there and y is copied back.
 * Both routes give the same bits. The caller keeps both host buffers allocated
 * and x_host unchanged until the stream has passed the call (kernels may still
 * be reading and writing them), and synchronizes the stream before reading
 * y_host.
 *   workspace_dev  device, >= zdmmv_host_step_workspace_bytes(rows, cols, batch),
 *                  16-byte aligned; holds x, its Q8_0 blocks and y (only the
 *                  Q8_0 blocks when the host buffers are used in place).
 * Errors: as zdmmv_q8_0_batched, plus ERR_SIZE. */
size_t zdmmv_host_step_workspace_bytes(int64_t rows, int64_t cols, int batch);
zdmmv_status zdmmv_host_step(zdmmv_fmt fmt, const void *w, zdmmv_layout layout,
                             int64_t rows, int64_t cols, const float *x_host, int batch,
                             float *y_host, void *workspace_dev, size_t workspace_bytes,
                             zdmmv_stream_t stream);

/* Debug / verification: the int32 per-block dot products s[r*nb+b] exactly as
 * the DMMV kernel that zdmmv_q{8,4}_0 would run for this shape forms them (same
 * device functions), for checking them bit for bit.
 *   sums  device int32 [rows][cols/32].
 * Errors: as zdmmv_q8_0, plus ERR_FORMAT. */
zdmmv_status zdmmv_debug_block_sums(zdmmv_fmt fmt, const void *w, zdmmv_layout layout,
                                    int64_t rows, int64_t cols, const void *xq,
                                    int32_t *sums, zdmmv_stream_t stream);

/* Self-test of the packed int8x4 dot on the device: out[i] = c[i] +
 * sum_j a[i].byte_j * b[i].byte_j (signed bytes), the "dp4a ... = 70" smoke of
 * "Bringing ZINC to NVIDIA", section "The reassuring result". All device
 * pointers, n >= 0 elements. Errors: ERR_NULL, ERR_SHAPE, ERR_CUDA. */
zdmmv_status zdmmv_selftest_dp4a(const int32_t *a, const int32_t *b, const int32_t *c,
                                 int32_t *out, int n, zdmmv_stream_t stream);

/* Self-test of the failure path: a kernel waits on a barrier that nothing ever
 * completes; the wait gives up after its bound (about 1 s), the kernel records
 * ZDMMV_FAULT_WAIT_TIMEOUT in the device fault word and stores 1 in result[0]
 * (0 would mean the wait completed), and returns normally -- no trap, no hang,
 * the context stays usable. result: device int32. Errors: ERR_NULL, ERR_CUDA. */
zdmmv_status zdmmv_selftest_wait_timeout(int32_t *result, zdmmv_stream_t stream);

/* Read (and, if clear != 0, reset) the device fault bits of the current device
 * (ZDMMV_FAULT_*). Synchronizes the device first. *bits_out = 0 means no kernel
 * has reported a fault. Errors: ERR_NULL, ERR_CUDA. */
zdmmv_status zdmmv_device_status(uint32_t *bits_out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* ZDMMV_H */
