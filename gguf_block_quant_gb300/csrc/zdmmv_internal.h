// zdmmv_internal.h -- host-side declarations shared by the translation units of
// libzdmmv.so (not part of the public C ABI; see include/zdmmv.h for that).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zdmmv {

// Arguments of the DMMV kernels (passed by value, like a push-constant block).
// One "slot" per blockIdx.y: slot k reads matrix w (+ idx[k]*expert_stride when
// idx is set), activation xq + k*xq_stride and writes y + k*y_stride.
struct DmmvArgs {
    const uint8_t *w;        // matrix base (GGUF blocks, or repacked quant stream + scales)
    const uint8_t *w_b;      // second stack (slots >= slots_a use it, with y_b), or nullptr
    float *y_b;              // output of the second stack's slot slots_a
    int32_t slots_a;         // slots of the first stack (when w_b is set)
    int64_t expert_stride;   // bytes between stacked matrices (gather)
    const int32_t *idx;      // device expert index per slot, or nullptr
    int32_t n_experts;       // valid index range [0, n_experts)
    int32_t *status;         // nullable: 1 is stored here for a bad index
    uint32_t *fault;         // device fault word (ZDMMV_FAULT_* bits)
    const uint8_t *xq;       // Q8_0 activation blocks of slot 0
    int64_t xq_stride;       // bytes between slots' activations (0 = shared)
    const float *xf;         // fp32 activation of slot 0 (fused-quantization kernels)
    int64_t xf_stride;       // floats between slots' fp32 activations
    float *y;                // output of slot 0
    int64_t y_stride;        // floats between slots' outputs
    int64_t rows;            // rows of the matrix
    int32_t nb;              // blocks per row
    int32_t batch;           // activation vectors per slot (plain kernel only)
    int32_t tile_rows;       // rows per pipeline stage (pipelined kernel)
    int32_t stage_bytes;     // shared-memory bytes per stage (pipelined kernel)
    int32_t x_bytes_padded;  // shared-memory bytes of the staged activation
    uint2 *argmax_parts;     // argmax epilogue: per-CTA (max bits, row), or nullptr
    const float *gate;       // accumulate epilogue: device scalar g, y += sigmoid(g) * W.x; nullptr: y += W.x
    int32_t accumulate;      // plain kernel: accumulate epilogue instead of store
    int32_t idx_ready;       // gather: the index list is complete when the grid starts (read before the wait)
};

// Most CTAs an argmax launch uses (its workspace holds one 8-byte partial each).
constexpr int kArgmaxMaxCtas = 2048;

// Launch description chosen by the host for the pipelined kernel.
struct TmaPlan {
    int lpr;         // lanes that share one row
    int ppl;         // block pairs per lane
    int stages;      // pipeline depth
    int tile_rows;   // rows per stage
    int stage_bytes;
    int x_bytes_padded;
    int smem_bytes;  // dynamic shared memory per CTA
};

constexpr int kConsumerThreads = 128;  // 4 consumer warps
constexpr int kProducerThreads = 32;   // 1 producer warp (one lane issues the copies)
constexpr int kTmaThreads = kConsumerThreads + kProducerThreads;
constexpr int kBarrierBytes = 256;     // shared-memory prefix holding the mbarriers
// CTAs of one pipelined launch per SM. A small launch takes fewer than fit (4 by
// registers and shared memory) on purpose: the free slots let the next decode
// kernel in the stream become resident and stream its weights while this one
// finishes (programmatic dependent launch). A large launch takes them all.
constexpr int kCtasPerSmSmall = 2;
constexpr int kCtasPerSmLarge = 4;
constexpr int64_t kLargeLaunchBytes = 32ll << 20;  // weight bytes per launch
constexpr int kSmemPerCtaTarget = 54 * 1024;         // keeps 4 CTAs per SM possible
constexpr int kTmaRowsIlp = 2;                       // rows per row group in flight

// Whether launches carry the programmatic-dependent-launch attribute (on unless
// the environment sets ZDMMV_PDL=0).
bool pdl_enabled();
// CTAs per SM a pipelined launch of this many weight bytes asks for (before the
// kernel's occupancy caps it); ZDMMV_CTAS_PER_SM (1..8) overrides it.
int ctas_per_sm_per_launch(int64_t weight_bytes, bool gathered = false);

// Allow a kernel the device's opt-in shared memory minus its static shared memory.
inline cudaError_t raise_dynamic_smem_limit(const void *fn, int dev) {
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - static_cast<int>(fa.sharedSizeBytes));
}

// Whether the pipelined kernel takes this shape, and its plan.
bool tma_shape_ok(int fmt, int64_t cols);
// unit_max_bytes: a tile of one pass of every row group with kTmaRowsIlp rows in
// flight is kept up to this size even above the stage target (single-vector
// launches: Q8_0 14336 x 4096 10.46 -> 10.0 us with 8-row tiles of 34.8 KB
// instead of 4-row ones; the vector split is slower with the larger tiles).
constexpr int kTmaWholeUnitMaxBytes = 40 * 1024;
TmaPlan tma_plan(int fmt, int layout, int64_t cols, int halves = 1, int unit_max_bytes = 0);

// Launchers of the pipelined kernel (one translation unit per format).
// fused_x: the kernel quantizes the fp32 activation a.xf itself (no a.xq).
cudaError_t launch_tma_q8(const DmmvArgs &a, const TmaPlan &p, int layout, bool fused_x, int ctas_per_slot,
                          int slots, cudaStream_t st, bool pdl);
cudaError_t launch_tma_q4(const DmmvArgs &a, const TmaPlan &p, int layout, bool fused_x, int ctas_per_slot,
                          int slots, cudaStream_t st, bool pdl);
// Batched kernel (one weight stream, 2..8 vectors): the plan and launchers.
struct BatchPlan {
    int g, bpt, vb;   // threads per row, blocks per thread, vectors per pass
    int stages, tile_rows, stage_bytes, x_bytes_padded, smem_bytes;
};
bool batch_plan(int fmt, int64_t cols, int batch, BatchPlan *out);
cudaError_t launch_batch_q8(const DmmvArgs &a, const BatchPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);
cudaError_t launch_batch_q4(const DmmvArgs &a, const BatchPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);

// The pipelined kernel with the argmax epilogue (no y written; per-CTA partials).
cudaError_t launch_argmax_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);
cudaError_t launch_argmax_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);

// The pipelined kernel with the accumulate epilogue (y += s * W.x).
cudaError_t launch_acc_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);
cudaError_t launch_acc_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl);

// The pipelined kernel with the SwiGLU pair epilogue (a.w gate, a.w_b up).
cudaError_t launch_swiglu_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                             cudaStream_t st, bool pdl);
cudaError_t launch_swiglu_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                             cudaStream_t st, bool pdl);
int swiglu_ctas_per_sm_q8(int layout, const TmaPlan &p);
int swiglu_ctas_per_sm_q4(int layout, const TmaPlan &p);

// Batched DMMV with the vectors split over the consumer warps: plan (false when
// the kernel does not take the shape and batch) and launchers.
bool vsplit_plan(int fmt, int layout, int64_t cols, int batch, TmaPlan *out, int *v, int *nvg);
cudaError_t launch_vsplit_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                             cudaStream_t st, bool pdl);
cudaError_t launch_vsplit_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                             cudaStream_t st, bool pdl);
// The same with the fp32 activations a.xf quantized in the kernel's prologue.
cudaError_t launch_vsplit_fx_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                                cudaStream_t st, bool pdl);
cudaError_t launch_vsplit_fx_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                                cudaStream_t st, bool pdl);

// The DMMV with an fp32 activation taken as is (no quantization): plan (false
// when the pipelined kernel does not take the shape) and launchers.
bool xf32_plan(int fmt, int layout, int64_t cols, TmaPlan *out);
cudaError_t launch_xf32_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                           cudaStream_t st, bool pdl);
cudaError_t launch_xf32_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                           cudaStream_t st, bool pdl);
cudaError_t launch_xf32_plain_q8(const DmmvArgs &a, int layout, int sms, int slots, cudaStream_t st, bool pdl);
cudaError_t launch_xf32_plain_q4(const DmmvArgs &a, int layout, int sms, int slots, cudaStream_t st, bool pdl);
// The tensor-core kernels' plans and launchers: zdmmv_mma.h.

// The one-launch expert FFN (gate/up + SwiGLU, then down): workspace size,
// shapes it takes, and the launcher (FfnArgs: zdmmv_ffn.cuh; the launcher fills
// in the plan fields).
struct FfnArgs;
size_t ffn_workspace_bytes(int n, int64_t ffn);
bool ffn_shape_ok(int fmt_gu, int fmt_dn, int64_t hidden, int64_t ffn);
cudaError_t launch_ffn(int fmt_gu, int fmt_dn, FfnArgs f, int sms, cudaStream_t st, bool pdl);
// The expert FFN entry point's checks and launch (status codes of zdmmv.h, as int).
int ffn_entry_status(int fmt_gu, const void *w_gate, const void *w_up, int64_t gu_stride, int fmt_dn,
                     const void *w_down, int64_t dn_stride, int64_t hidden, int64_t ffn, const int32_t *idx, int n,
                     int n_experts, const void *xq, float *y, void *workspace, size_t workspace_bytes,
                     int32_t *status_dev, cudaStream_t st, bool pdl);

// The argmax DMMV (per-CTA partials at `parts`, room for kArgmaxMaxCtas) and its
// one-CTA reduce, on the current device; arguments already checked. Shared by the
// workspace and the allocation-free argmax entry points.
cudaError_t launch_argmax_dmmv(int fmt, int layout, const void *w, int64_t rows, int64_t cols, const void *xq,
                               int32_t *argmax_out, float *max_out, uint2 *parts, cudaStream_t st);
// The argmax epilogue's final pass (one CTA over n partials).
cudaError_t launch_argmax_reduce(const uint2 *parts, int n, int32_t *argmax_out, float *max_out, cudaStream_t st,
                                 bool pdl);
// The device fault word of the current device (nullptr on error).
uint32_t *current_fault_word();

// CTAs of the pipelined kernel that fit on one SM for this plan.
int tma_ctas_per_sm_q8(int layout, const TmaPlan &p);
int tma_ctas_per_sm_q4(int layout, const TmaPlan &p);

}  // namespace zdmmv
