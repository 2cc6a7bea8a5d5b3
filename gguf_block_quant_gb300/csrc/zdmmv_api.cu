// zdmmv_api.cu -- the C ABI of libzdmmv.so: argument checks, launch planning and
// the small kernels (activation quantizer, repack, plain DMMV, debug sums, dp4a
// self-test). The TMA-pipelined DMMV kernels live in zdmmv_tma_q8.cu /
// zdmmv_tma_q4.cu. The library allocates no device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "zdmmv.h"
#include "zdmmv_device.cuh"
#include "zdmmv_internal.h"
#include "zdmmv_mma.h"
#include "zdmmv_xf32_mma.cuh"
#include "zdmmv_bmma.cuh"

namespace zdmmv {

// ------------------------------------------------------------- fault word
// One word per device that kernels OR fault bits into (bounded waits that gave
// up). Read and cleared by zdmmv_device_status.
__device__ uint32_t g_fault_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    uint32_t *fault = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mu;

cudaError_t device_info(const DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fault_word);
        if (e != cudaSuccess) return e;
        d.fault = static_cast<uint32_t *>(p);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

}  // namespace

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("ZDMMV_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

// CTAs of one pipelined launch per SM: kCtasPerSmSmall below kLargeLaunchBytes
// of weights, kCtasPerSmLarge above. A gathered launch (expert indices read on
// the device) cannot stream any weights before its dependency wait, so it takes
// as many CTAs as fit, for more requests in flight once it may start (measured
// on the MoE step: gate+up 9.3 -> 7.7 us from 2 to 5 CTAs per SM). The
// environment variable ZDMMV_CTAS_PER_SM (1..8) overrides all three.
constexpr int kCtasPerSmGathered = 8;  // capped by the occupancy of the kernel
int ctas_per_sm_per_launch(int64_t weight_bytes, bool gathered) {
    static const int forced = [] {
        const char *e = std::getenv("ZDMMV_CTAS_PER_SM");
        const int n = e ? std::atoi(e) : 0;
        return (n >= 1 && n <= 8) ? n : 0;
    }();
    if (forced) return forced;
    if (gathered) return kCtasPerSmGathered;
    return weight_bytes >= kLargeLaunchBytes ? kCtasPerSmLarge : kCtasPerSmSmall;
}

namespace {

// Batched calls stream the weights once (dmmv_batch_kernel) unless
// ZDMMV_BATCH_SLOTS=1, which runs one single-vector slot per vector instead.
int batch_slots_forced() {
    static const int v = [] {
        const char *e = std::getenv("ZDMMV_BATCH_SLOTS");
        return (e && e[0] == '1') ? 1 : 0;
    }();
    return v;
}

// CTAs per SM of a batched launch (environment ZDMMV_BATCH_CTAS_PER_SM, 1..4; default 2)
int batch_ctas_per_sm() {
    static const int v = [] {
        const char *e = std::getenv("ZDMMV_BATCH_CTAS_PER_SM");
        const int n = e ? std::atoi(e) : 0;
        return (n >= 1 && n <= 4) ? n : 3;
    }();
    return v;
}

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline int block_bytes(int fmt) { return fmt == kFmtQ8 ? 34 : (fmt == kFmtQ4 ? 18 : 0); }
inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

zdmmv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ZDMMV_OK : ZDMMV_ERR_CUDA; }

// Launch without attributes; the launch's own error is returned (never an
// earlier one left behind by an unrelated call).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain_cfg(void (*kern)(KArgs...), unsigned grid, unsigned block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

// ------------------------------------------------------------ planning
namespace {
// Target bytes of one pipeline stage (environment ZDMMV_STAGE_KB, 4..64).
int stage_target_bytes() {
    static const int v = [] {
        const char *e = std::getenv("ZDMMV_STAGE_KB");
        const int n = e ? std::atoi(e) : 0;
        return (n >= 4 && n <= 64 ? n : 20) * 1024;
    }();
    return v;
}
}  // namespace

bool tma_shape_ok(int fmt, int64_t cols) {
    if (block_bytes(fmt) == 0 || cols <= 0 || cols % kQK) return false;
    const int64_t nb = cols / kQK;
    // rows must be 16-byte multiples (bulk copies) and the activation must fit
    // the register budget: at most 4 pairs per lane with 32 lanes per row
    return nb % 8 == 0 && nb / 2 <= 128;
}

TmaPlan tma_plan(int fmt, int layout, int64_t cols, int halves, int unit_max_bytes) {
    (void)layout;
    TmaPlan p{};
    const int nb = static_cast<int>(cols / kQK);
    const int npairs = nb / 2;
    if (npairs <= 8) {
        p.lpr = 8; p.ppl = 1;
    } else if (npairs <= 16) {
        p.lpr = 16; p.ppl = 1;
    } else if (npairs <= 32) {
        p.lpr = 32; p.ppl = 1;
    } else if (npairs <= 64) {
        p.lpr = 32; p.ppl = 2;
    } else {
        p.lpr = 32; p.ppl = 4;
    }
    const int rows_par = kConsumerThreads / p.lpr;
    const int row_bytes = nb * block_bytes(fmt);
    // a pair stage (halves = 2) holds the same rows of two matrices
    const int stage_target = stage_target_bytes() / halves;
    // a tile is a whole number of passes of the row groups (kTmaRowsIlp rows each
    // when that fits the stage target, or unit_max_bytes where the caller allows
    // more)
    int unit_rows = rows_par * kTmaRowsIlp;
    const int unit_cap = unit_max_bytes > stage_target ? unit_max_bytes : stage_target;
    if (unit_rows * row_bytes > unit_cap) unit_rows = rows_par;
    const int unit = unit_rows * row_bytes;
    const int m = unit >= stage_target ? 1 : stage_target / unit;
    p.tile_rows = unit_rows * m;
    p.stage_bytes = halves * static_cast<int>(round_up(static_cast<int64_t>(p.tile_rows) * row_bytes, 128));
    p.x_bytes_padded = static_cast<int>(round_up(static_cast<int64_t>(nb) * 34, 128));
    p.stages = 4;
    while (p.stages > 2 && kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes > kSmemPerCtaTarget)
        --p.stages;
    p.smem_bytes = kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes;
    return p;
}

namespace {
// Batched kernel choice (environment ZDMMV_BATCH_KERNEL). Unset: the fp16
// tensor-core kernel for kBmmaMinBatch..8 vectors where it takes the shape and
// has a 32-row group for every SM, else the vector split, else the streaming
// batch kernel. "vsplit": never the tensor-core kernel. "mma": the tensor-core
// kernel wherever it takes the shape (2..8 vectors). "stream": dmmv_batch_kernel.
// "slots": single-vector slots (as ZDMMV_BATCH_SLOTS=1).
enum BatchChoice { kBatchAuto = 0, kBatchStream = 1, kBatchSlots = 2, kBatchMma = 3, kBatchVsplit = 4 };
// From 5 vectors on the vector split is bound by its dp4a issue (Q8_0 14336 x
// 4096: 10.8 / 11.8 / 15.2 / 15.3 us at 2 / 4 / 5 / 8 vectors) and the
// tensor-core kernel is faster (12.7 us at any batch).
constexpr int kBmmaMinBatch = 5;
int batch_kernel_choice() {
    static const int v = [] {
        const char *e = std::getenv("ZDMMV_BATCH_KERNEL");
        if (!e) return static_cast<int>(kBatchAuto);
        if (std::strcmp(e, "stream") == 0) return static_cast<int>(kBatchStream);
        if (std::strcmp(e, "slots") == 0) return static_cast<int>(kBatchSlots);
        if (std::strcmp(e, "mma") == 0) return static_cast<int>(kBatchMma);
        if (std::strcmp(e, "vsplit") == 0) return static_cast<int>(kBatchVsplit);
        return static_cast<int>(kBatchAuto);
    }();
    return v;
}
// Vectors per warp in the vector-split kernel for batches above 2 (environment
// ZDMMV_VSPLIT_V=1 forces one; the default takes two where the registers allow).
int vsplit_v_pref() {
    static const int v = [] {
        const char *e = std::getenv("ZDMMV_VSPLIT_V");
        return (e && std::atoi(e) == 1) ? 1 : 2;
    }();
    return v;
}
}  // namespace

bool vsplit_plan(int fmt, int layout, int64_t cols, int batch, TmaPlan *out, int *v, int *nvg) {
    if (!tma_shape_ok(fmt, cols) || batch < 2 || batch > ZDMMV_MAX_BATCH) return false;
    TmaPlan p = tma_plan(fmt, layout, cols);
    // one vector per warp for two vectors (two row groups of warps each); two
    // per warp beyond, while their block-pair registers fit (at most 2 pairs per lane)
    const int vv = (batch > 2 && p.ppl <= 2 && vsplit_v_pref() == 2) ? 2 : 1;
    const int groups = (batch + vv - 1) / vv;
    const int ng = groups <= 1 ? 1 : (groups <= 2 ? 2 : (groups <= 4 ? 4 : 0));
    if (ng == 0 || (vv == 1 && ng == 1)) return false;
    // the batch's activation blocks are staged once; 3 stages when three CTAs
    // per SM still fit, else 2
    p.x_bytes_padded = static_cast<int>(round_up(static_cast<int64_t>(batch) * (cols / kQK) * 34, 128));
    p.stages = kBarrierBytes + p.x_bytes_padded + 3 * p.stage_bytes <= 72 * 1024 ? 3 : 2;
    p.smem_bytes = kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes;
    *out = p;
    *v = vv;
    *nvg = ng;
    return true;
}

bool xf32_plan(int fmt, int layout, int64_t cols, TmaPlan *out) {
    (void)layout;
    if (!tma_shape_ok(fmt, cols)) return false;
    const int nb = static_cast<int>(cols / kQK);
    TmaPlan p{};
    p.lpr = nb % 32 == 0 ? 32 : (nb % 16 == 0 ? 16 : 8);
    const int rows_par = kConsumerThreads / p.lpr;
    const int row_bytes = nb * block_bytes(fmt);
    // Prefer a plan that leaves room for 4 CTAs per SM (the kernel is bound by
    // its fp32 arithmetic, so resident warps matter more than deep pipelining);
    // wide rows fall back to larger units and 2 CTAs per SM.
    const int x_bytes = static_cast<int>(round_up(static_cast<int64_t>(nb) * 144, 128));
    const int small_budget = 56 * 1024 - kBarrierBytes - x_bytes;
    const int kUnitMax = small_budget >= 2 * 12 * 1024 ? small_budget / 2 : 36 * 1024;
    const int kStageTarget = kUnitMax;
    p.ppl = 0;
    for (int r = 4; r >= 1; r >>= 1)
        if (rows_par * r * row_bytes <= kUnitMax) {
            p.ppl = r;
            break;
        }
    if (p.ppl == 0) return false;
    const int unit_rows = rows_par * p.ppl;
    const int unit = unit_rows * row_bytes;
    const int m = unit >= kStageTarget ? 1 : kStageTarget / unit;
    p.tile_rows = unit_rows * m;
    p.stage_bytes = static_cast<int>(round_up(static_cast<int64_t>(p.tile_rows) * row_bytes, 128));
    p.x_bytes_padded = x_bytes;
    p.stages = kBarrierBytes + p.x_bytes_padded + 3 * p.stage_bytes <= 56 * 1024 ? 3 : 2;
    p.smem_bytes = kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes;
    if (p.smem_bytes > 112 * 1024) return false;
    *out = p;
    return true;
}

bool batch_plan(int fmt, int64_t cols, int batch, BatchPlan *out) {
    if (!tma_shape_ok(fmt, cols) || batch < 2 || batch > ZDMMV_MAX_BATCH) return false;
    const int nb = static_cast<int>(cols / kQK);
    BatchPlan p{};
    if (nb % 128 == 0 && nb / 128 <= 2) {
        p.g = 128; p.bpt = nb / 128;
    } else if (nb == 64) {
        p.g = 64; p.bpt = 1;
    } else if (nb % 32 == 0 && nb / 32 <= 4) {
        p.g = 32; p.bpt = nb / 32;
    } else {
        return false;  // other widths take the per-vector slots of the single-vector kernel
    }
    // vectors held in registers per pass: all of them with one block per thread
    if (p.bpt == 1)
        p.vb = batch <= 2 ? 2 : (batch <= 4 ? 4 : 8);
    else
        p.vb = p.bpt == 2 ? 2 : 1;
    const int groups = kConsumerThreads / p.g;
    const int row_bytes = nb * block_bytes(fmt);
    const int unit_rows = groups * 2;  // two rows per group per iteration
    const int stage_target = stage_target_bytes();
    const int unit = unit_rows * row_bytes;
    const int m = unit >= stage_target ? 1 : stage_target / unit;
    p.tile_rows = unit_rows * m;
    p.stage_bytes = static_cast<int>(round_up(static_cast<int64_t>(p.tile_rows) * row_bytes, 128));
    p.x_bytes_padded = 0;  // each thread loads its activation blocks straight into registers
    // per-tile partial sums: [passes][iterations][groups][warps per group][2*vb] floats
    const int npass = (batch + p.vb - 1) / p.vb;
    const int iters = (p.tile_rows + unit_rows - 1) / unit_rows;
    const int red_bytes = npass * iters * (kConsumerThreads / 32) * 2 * p.vb * 4;
    p.stages = 4;
    while (p.stages > 2 &&
           kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes + red_bytes > kSmemPerCtaTarget)
        --p.stages;
    p.smem_bytes = kBarrierBytes + p.x_bytes_padded + p.stages * p.stage_bytes + red_bytes;
    if (p.smem_bytes > 200 * 1024) return false;
    *out = p;
    return true;
}

// ------------------------------------------------------------- kernels
__device__ __forceinline__ void pdl_wait_api() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger_api() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One warp per Q8_0 block: lane j owns element j.
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float *__restrict__ x, int64_t nblocks,
                                                            uint8_t *__restrict__ xq) {
    pdl_wait_api();
    pdl_trigger_api();
    const int lane = threadIdx.x & 31;
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= nblocks) return;
    const float v = x[blk * kQK + lane];
    unsigned short d_bits;
    const int q = quantize_q8_0_lane(v, d_bits);
    uint8_t *out = xq + blk * 34;
    out[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    if (lane == 0) *reinterpret_cast<unsigned short *>(out) = d_bits;  // one 2-byte store (blocks are 2-byte aligned)
}

// One thread per block: GGUF block -> quant stream slot + scale slot.
template <int FMT>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ src, int64_t nblocks,
                                                     uint8_t *__restrict__ dst) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const uint16_t *h = reinterpret_cast<const uint16_t *>(src + i * kBB);
    uint32_t q[kQB / 4];
#pragma unroll
    for (int k = 0; k < kQB / 4; ++k) q[k] = ld_u16_pair(h + 1 + 2 * k);
    uint4 *dq = reinterpret_cast<uint4 *>(dst + i * kQB);
#pragma unroll
    for (int k = 0; k < kQB / 16; ++k) dq[k] = make_uint4(q[4 * k], q[4 * k + 1], q[4 * k + 2], q[4 * k + 3]);
    reinterpret_cast<uint16_t *>(dst + nblocks * kQB)[i] = h[0];
}

// Final pass of the argmax epilogue: one CTA reduces the per-CTA partials with
// the same ordering (larger value, then smaller row).
__global__ void __launch_bounds__(256) argmax_reduce_kernel(const uint2 *__restrict__ parts, int n,
                                                            int32_t *__restrict__ out_row, float *__restrict__ out_max) {
    pdl_wait_api();
    pdl_trigger_api();
    __shared__ float sv[8];
    __shared__ int sr[8];
    float bv = 0.0f;
    int br = -1;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const uint2 p = parts[i];
        const float v = __uint_as_float(p.x);
        const int r = static_cast<int>(p.y);
        if (r >= 0 && (br < 0 || v > bv || (v == bv && r < br))) {
            bv = v;
            br = r;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, bv, o);
        const int r = __shfl_xor_sync(0xffffffffu, br, o);
        if (r >= 0 && (br < 0 || v > bv || (v == bv && r < br))) {
            bv = v;
            br = r;
        }
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sv[warp] = bv;
        sr[warp] = br;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int q = 1; q < static_cast<int>(blockDim.x >> 5); ++q)
            if (sr[q] >= 0 && (br < 0 || sv[q] > bv || (sv[q] == bv && sr[q] < br))) {
                bv = sv[q];
                br = sr[q];
            }
        out_row[0] = br;
        if (out_max) out_max[0] = bv;
    }
}

// Failure-path self-test: one warp waits on an mbarrier that nothing ever
// completes. The bounded wait gives up, the fault bit is recorded and
// result[0] = 1; the kernel then returns normally.
__global__ void selftest_wait_timeout_kernel(uint32_t *fault, int32_t *result) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrival that never comes
        fence_barrier_init();
    }
    __syncwarp();
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bar, 0));
    if (threadIdx.x == 0) {
        if (!done) atomicOr(fault, ZDMMV_FAULT_WAIT_TIMEOUT);
        result[0] = done ? 0 : 1;
    }
}

__global__ void selftest_dp4a_kernel(const int32_t *a, const int32_t *b, const int32_t *c, int32_t *out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = dp4a_ss(static_cast<uint32_t>(a[i]), static_cast<uint32_t>(b[i]), c[i]);
}

// Plain DMMV for the shapes the pipelined kernel does not take (rows that are
// not 16-byte multiples, very long rows): one warp per row, lanes stride over
// blocks with 16-bit loads. Same block arithmetic, fp32 accumulation and
// xor-shuffle reduction. Handles `batch` vectors per slot and expert slots.
template <int FMT, int LAYOUT>
__global__ void __launch_bounds__(256) dmmv_plain_kernel(const DmmvArgs a) {
    pdl_wait_api();
    pdl_trigger_api();
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int slot = blockIdx.y;
    if (row >= a.rows) return;
    const bool second = a.w_b != nullptr && slot >= a.slots_a;
    const int sel = second ? slot - a.slots_a : slot;
    float *y = (second ? a.y_b : a.y) + sel * a.y_stride;
    const uint8_t *w = second ? a.w_b : a.w;
    if (a.idx != nullptr) {
        const int e = a.idx[sel];
        if (e < 0 || e >= a.n_experts) {
            if (lane == 0) {
                y[row] = __int_as_float(0x7fc00000);
                if (a.status != nullptr) atomicExch(a.status, 1);
            }
            return;
        }
        w += static_cast<int64_t>(e) * a.expert_stride;
    }
    const int nb = a.nb;
    const uint8_t *xq0 = a.xq + sel * a.xq_stride;
    for (int v = 0; v < a.batch; ++v) {
        const uint8_t *xq = xq0 + static_cast<int64_t>(v) * nb * 34;
        float acc = 0.0f;
        for (int b = lane; b < nb; b += 32) {
            uint32_t q[8], xw[8];
            float dw, dx;
            const int64_t blk = row * nb + b;
            if constexpr (LAYOUT == kLayoutGguf)
                Block<FMT>::load_gguf(w + blk * kBB, q, dw);
            else
                Block<FMT>::load_repacked(w + blk * kQB, w + a.rows * nb * kQB + blk * 2, q, dw);
            load_x_block(xq + static_cast<int64_t>(b) * 34, xw, dx);
            const int s = Block<FMT>::dot(q, xw);
            acc = __fmaf_rn(static_cast<float>(s), __fmul_rn(dw, dx), acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            float *dst = y + static_cast<int64_t>(v) * a.rows + row;
            if (a.accumulate) {
                const float scale = a.gate != nullptr ? 1.0f / (1.0f + expf(-*a.gate)) : 1.0f;
                *dst = __fmaf_rn(scale, acc, *dst);
            } else {
                *dst = acc;
            }
        }
    }
}

// Plain DMMV with the fp32 activation quantized by each CTA into shared memory
// first (same quantizer device function as everywhere else), then one warp per
// row over a grid-stride row loop. Used by the fused entry point for shapes the
// pipelined kernel does not take.
template <int FMT, int LAYOUT>
__global__ void __launch_bounds__(256) dmmv_plain_fx_kernel(const DmmvArgs a) {
    extern __shared__ __align__(16) uint8_t xsm[];  // batch * nb Q8_0 blocks
    pdl_wait_api();
    pdl_trigger_api();
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nb = a.nb;
    const int total = a.batch * nb;
    for (int b = warp; b < total; b += nwarps) {
        const int v = b / nb;
        const int blk = b - v * nb;
        const float xv = a.xf[static_cast<int64_t>(v) * a.xf_stride + static_cast<int64_t>(blk) * kQK + lane];
        unsigned short d_bits;
        const int q = quantize_q8_0_lane(xv, d_bits);
        xsm[34 * b + 2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
        if (lane == 0) *reinterpret_cast<unsigned short *>(xsm + 34 * b) = d_bits;
    }
    __syncthreads();
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * nwarps + warp; row < a.rows;
         row += static_cast<int64_t>(gridDim.x) * nwarps) {
        for (int v = 0; v < a.batch; ++v) {
            const uint8_t *xq = xsm + static_cast<int64_t>(v) * nb * 34;
            float acc = 0.0f;
            for (int b = lane; b < nb; b += 32) {
                uint32_t q[8], xw[8];
                float dw, dx;
                const int64_t blk = row * nb + b;
                if constexpr (LAYOUT == kLayoutGguf)
                    Block<FMT>::load_gguf(a.w + blk * kBB, q, dw);
                else
                    Block<FMT>::load_repacked(a.w + blk * kQB, a.w + a.rows * nb * kQB + blk * 2, q, dw);
                load_x_block(xq + static_cast<int64_t>(b) * 34, xw, dx);
                const int s = Block<FMT>::dot(q, xw);
                acc = __fmaf_rn(static_cast<float>(s), __fmul_rn(dw, dx), acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) a.y[static_cast<int64_t>(v) * a.rows + row] = acc;
        }
    }
}

// Debug: the int32 block sums with the device functions of the kernel that the
// DMMV entry points pick for this shape. PAIRS: one thread per (row, pair) via
// Pair<>::sums (pipelined kernel); else one thread per (row, block) via Block<>.
template <int FMT, int LAYOUT, bool PAIRS>
__global__ void __launch_bounds__(256) block_sums_kernel(const uint8_t *__restrict__ w, int64_t rows, int nb,
                                                         const uint8_t *__restrict__ xq, int32_t *__restrict__ sums) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if constexpr (PAIRS) {
        const int npairs = nb / 2;
        if (t >= rows * npairs) return;
        const int64_t row = t / npairs;
        const int p = static_cast<int>(t % npairs);
        uint32_t v[17];
        load_x_pair_words(xq, p, v);
        Pair<FMT, LAYOUT> pr;
        pr.set(v);
        constexpr int kW = Pair<FMT, LAYOUT>::kWords;
        uint32_t ww[kW];
        const uint32_t *src;
        if constexpr (LAYOUT == kLayoutGguf)
            src = reinterpret_cast<const uint32_t *>(w + row * nb * kBB + static_cast<int64_t>(p) * 2 * kBB);
        else
            src = reinterpret_cast<const uint32_t *>(w + (row * nb + 2 * p) * kQB);
#pragma unroll
        for (int k = 0; k < kW; ++k) ww[k] = src[k];
        int sa, sb;
        pr.sums(ww, sa, sb);
        sums[row * nb + 2 * p] = sa;
        sums[row * nb + 2 * p + 1] = sb;
    } else {
        if (t >= rows * nb) return;
        const int b = static_cast<int>(t % nb);
        uint32_t q[8], xw[8];
        float dw, dx;
        if constexpr (LAYOUT == kLayoutGguf)
            Block<FMT>::load_gguf(w + t * kBB, q, dw);
        else
            Block<FMT>::load_repacked(w + t * kQB, w + rows * nb * kQB + t * 2, q, dw);
        load_x_block(xq + static_cast<int64_t>(b) * 34, xw, dx);
        sums[t] = Block<FMT>::dot(q, xw);
    }
}

// --------------------------------------------------------- launch helpers
namespace {

cudaError_t launch_plain(int fmt, int layout, const DmmvArgs &a, int slots, cudaStream_t st) {
    if (a.rows == 0 || slots == 0) return cudaSuccess;
    const int64_t blocks = (a.rows + 7) / 8;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(slots), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (fmt == kFmtQ8)
        return layout == kLayoutGguf ? cudaLaunchKernelEx(&cfg, dmmv_plain_kernel<kFmtQ8, kLayoutGguf>, a)
                                     : cudaLaunchKernelEx(&cfg, dmmv_plain_kernel<kFmtQ8, kLayoutRepacked>, a);
    return layout == kLayoutGguf ? cudaLaunchKernelEx(&cfg, dmmv_plain_kernel<kFmtQ4, kLayoutGguf>, a)
                                 : cudaLaunchKernelEx(&cfg, dmmv_plain_kernel<kFmtQ4, kLayoutRepacked>, a);
}

constexpr int kPlainFxMaxSmem = 200 * 1024;

cudaError_t launch_plain_fx(int fmt, int layout, const DmmvArgs &a, int sms, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(a.batch) * a.nb * 34;
    int64_t ctas = (a.rows + 7) / 8;
    if (ctas > static_cast<int64_t>(sms) * 4) ctas = static_cast<int64_t>(sms) * 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    auto go = [&](auto kern) -> cudaError_t {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kern), dev);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, kern, a);
    };
    if (fmt == kFmtQ8)
        return layout == kLayoutGguf ? go(dmmv_plain_fx_kernel<kFmtQ8, kLayoutGguf>)
                                     : go(dmmv_plain_fx_kernel<kFmtQ8, kLayoutRepacked>);
    return layout == kLayoutGguf ? go(dmmv_plain_fx_kernel<kFmtQ4, kLayoutGguf>)
                                 : go(dmmv_plain_fx_kernel<kFmtQ4, kLayoutRepacked>);
}

// Run the DMMV over `slots` slots (expert gather / batch through slots).
// fused_x: the activation is fp32 (a.xf) and the kernel quantizes it itself.
zdmmv_status run_dmmv(int fmt, int layout, DmmvArgs a, int slots, cudaStream_t st, bool fused_x = false) {
    const DeviceInfo *dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return ZDMMV_ERR_CUDA;
    a.fault = dev->fault;
    if (a.rows == 0 || slots == 0) return ZDMMV_OK;
    const int64_t cols = static_cast<int64_t>(a.nb) * kQK;
    if (tma_shape_ok(fmt, cols) && a.batch == 1) {
        const TmaPlan p = tma_plan(fmt, layout, cols, 1, kTmaWholeUnitMaxBytes);
        a.tile_rows = p.tile_rows;
        a.stage_bytes = p.stage_bytes;
        a.x_bytes_padded = p.x_bytes_padded;
        int per_sm = fmt == kFmtQ8 ? tma_ctas_per_sm_q8(layout, p) : tma_ctas_per_sm_q4(layout, p);
        const int64_t launch_bytes = a.rows * a.nb * static_cast<int64_t>(block_bytes(fmt)) * slots;
        // a gather that reads its indices before the dependency wait streams its
        // weights early like a plain DMMV and takes the plain launch's CTAs per SM
        // (MoE down gather after gate/up: 2 per SM 7.15 us per token-layer, as many
        // as fit 7.29 us)
        const int want = ctas_per_sm_per_launch(launch_bytes, a.idx != nullptr && !a.idx_ready);
        if (per_sm > want) per_sm = want;
        const int64_t total = static_cast<int64_t>(dev->sms) * per_sm;
        int64_t ctas = total / slots;
        if (ctas < 1) ctas = 1;
        if (ctas > a.rows) ctas = a.rows;
        if (ctas > 65535) ctas = 65535;
        e = fmt == kFmtQ8
                ? launch_tma_q8(a, p, layout, fused_x, static_cast<int>(ctas), slots, st, pdl_enabled())
                : launch_tma_q4(a, p, layout, fused_x, static_cast<int>(ctas), slots, st, pdl_enabled());
        return from_cuda(e);
    }
    if (fused_x) return from_cuda(launch_plain_fx(fmt, layout, a, dev->sms, st));
    return from_cuda(launch_plain(fmt, layout, a, slots, st));
}

zdmmv_status check_matrix(int fmt, const void *w, int layout, int64_t rows, int64_t cols, const void *xq,
                          const float *y) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    if (rows < 0 || cols <= 0 || cols % kQK) return ZDMMV_ERR_SHAPE;
    if (cols / kQK > 0x3fffffff) return ZDMMV_ERR_SHAPE;
    if (rows == 0) return ZDMMV_OK;
    if (!w || !xq || !y) return ZDMMV_ERR_NULL;
    if (!aligned(w, 16) || !aligned(xq, 16) || !aligned(y, 4)) return ZDMMV_ERR_ALIGN;
    return ZDMMV_OK;
}

zdmmv_status dmmv_entry(int fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols, const void *xq,
                        int batch, float *y, cudaStream_t st) {
    zdmmv_status s = check_matrix(fmt, w, layout, rows, cols, xq, y);
    if (s != ZDMMV_OK) return s;
    if (batch < 1 || batch > ZDMMV_MAX_BATCH) return ZDMMV_ERR_SHAPE;
    if (rows == 0) return ZDMMV_OK;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.y = y;
    a.rows = rows;
    a.nb = static_cast<int32_t>(cols / kQK);
    BatchPlan bp{};
    TmaPlan vp{};
    int vv = 0, nvg = 0;
    const int choice = batch_slots_forced() ? kBatchSlots : batch_kernel_choice();
    BmmaPlan hp{};
    if (batch >= 2 && (choice == kBatchMma || (choice == kBatchAuto && batch >= kBmmaMinBatch)) &&
        bmma_plan(fmt, layout, rows, cols, batch, &hp)) {
        // one weight stream, all vectors on the fp16 tensor cores (by default only
        // where every SM gets a 32-row group: on fewer rows the vector split's
        // finer row split keeps more SMs streaming)
        const DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
        if (choice == kBatchMma || (rows + kBmGroupRows - 1) / kBmGroupRows >= dev->sms) {
            BmmaArgs m{};
            m.w = a.w;
            m.xq = a.xq;
            m.y = y;
            m.fault = dev->fault;
            m.rows = rows;
            m.xq_stride = static_cast<int64_t>(a.nb) * 34;
            m.y_stride = rows;
            m.nb = a.nb;
            m.batch = batch;
            m.nchunks = hp.nchunks;
            m.pitch = hp.pitch;
            m.red_bufs = hp.red_bufs;
            return from_cuda(launch_bmma(fmt, m, hp, false, st, pdl_enabled()));
        }
    }
    if (batch >= 2 && (choice == kBatchAuto || choice == kBatchMma || choice == kBatchVsplit) &&
        vsplit_plan(fmt, layout, cols, batch, &vp, &vv, &nvg)) {
        // one weight stream, the vectors split over the warps
        const DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
        a.fault = dev->fault;
        a.batch = batch;
        a.xq_stride = static_cast<int64_t>(a.nb) * 34;
        a.y_stride = rows;
        a.tile_rows = vp.tile_rows;
        a.stage_bytes = vp.stage_bytes;
        a.x_bytes_padded = vp.x_bytes_padded;
        const int cap = std::getenv("ZDMMV_BATCH_CTAS_PER_SM") ? batch_ctas_per_sm() : 0;
        cudaError_t e = fmt == kFmtQ8 ? launch_vsplit_q8(a, vp, layout, vv, nvg, cap, st, pdl_enabled())
                                      : launch_vsplit_q4(a, vp, layout, vv, nvg, cap, st, pdl_enabled());
        return from_cuda(e);
    }
    if (batch >= 2 && choice != kBatchSlots && batch_plan(fmt, cols, batch, &bp)) {
        // one weight stream for all vectors
        const DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
        a.fault = dev->fault;
        a.batch = batch;
        a.y_stride = rows;
        a.tile_rows = bp.tile_rows;
        a.stage_bytes = bp.stage_bytes;
        a.x_bytes_padded = bp.x_bytes_padded;
        int64_t ctas = static_cast<int64_t>(dev->sms) * batch_ctas_per_sm();
        if (ctas > rows) ctas = rows;
        cudaError_t e = fmt == kFmtQ8 ? launch_batch_q8(a, bp, layout, static_cast<int>(ctas), st, pdl_enabled())
                                      : launch_batch_q4(a, bp, layout, static_cast<int>(ctas), st, pdl_enabled());
        return from_cuda(e);
    }
    if (tma_shape_ok(fmt, cols)) {
        // batch vectors as slots of the pipelined kernel: slot v reads
        // activation v and writes output row block v
        a.batch = 1;
        a.xq_stride = static_cast<int64_t>(a.nb) * 34;
        a.y_stride = rows;
        return run_dmmv(fmt, layout, a, batch, st);
    }
    a.batch = batch;
    return run_dmmv(fmt, layout, a, 1, st);
}

zdmmv_status gather_entry(int fmt, const void *w_stack, const void *w_stack_b, int64_t expert_stride_bytes,
                          int layout, int64_t rows, int64_t cols, const int32_t *idx, int n, int n_experts,
                          const void *xq, int64_t xq_stride_bytes, float *y, float *y_b, int32_t *status_dev,
                          cudaStream_t st, bool idx_ready = false) {
    zdmmv_status s = check_matrix(fmt, w_stack, layout, rows, cols, xq, y);
    if (s != ZDMMV_OK) return s;
    if (n < 0 || n > 32767 || n_experts < 0) return ZDMMV_ERR_SHAPE;
    if (n == 0 || rows == 0) return ZDMMV_OK;
    if (!idx) return ZDMMV_ERR_NULL;
    if (!aligned(idx, 4) || (status_dev && !aligned(status_dev, 4))) return ZDMMV_ERR_ALIGN;
    if (w_stack_b && (!aligned(w_stack_b, 16) || !aligned(y_b, 4))) return ZDMMV_ERR_ALIGN;
    const int64_t nb = cols / kQK;
    const int64_t mat_bytes = rows * nb * block_bytes(fmt);
    if (expert_stride_bytes < 0 || xq_stride_bytes < 0) return ZDMMV_ERR_SHAPE;
    if (n_experts > 1 && expert_stride_bytes < mat_bytes) return ZDMMV_ERR_SHAPE;
    if (xq_stride_bytes != 0 && xq_stride_bytes < nb * 34) return ZDMMV_ERR_SHAPE;
    if (expert_stride_bytes % 16 || xq_stride_bytes % 16) return ZDMMV_ERR_ALIGN;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w_stack);
    a.w_b = static_cast<const uint8_t *>(w_stack_b);
    a.y_b = y_b;
    a.slots_a = n;
    a.expert_stride = expert_stride_bytes;
    a.idx = idx;
    a.n_experts = n_experts;
    a.status = status_dev;
    a.xq = static_cast<const uint8_t *>(xq);
    a.xq_stride = xq_stride_bytes;
    a.y = y;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(nb);
    a.batch = 1;
    a.idx_ready = idx_ready ? 1 : 0;
    return run_dmmv(fmt, layout, a, w_stack_b ? 2 * n : n, st);
}

// Expert gather over fp32 activations: the pipelined kernel's fused-quantization
// variant with one slot per selected expert (each CTA quantizes its slot's
// activation with the stand-alone quantizer's arithmetic, so the result is the
// quantizer followed by the gather, bit for bit).
zdmmv_status gather_f32_entry(int fmt, const void *w_stack, int64_t expert_stride_bytes, int layout, int64_t rows,
                              int64_t cols, const int32_t *idx, int n, int n_experts, const float *x,
                              int64_t x_stride, float *y, int32_t *status_dev, bool idx_ready, cudaStream_t st) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    if (rows < 0 || cols <= 0 || cols % kQK || n < 0 || n > 32767 || n_experts < 0) return ZDMMV_ERR_SHAPE;
    if (n == 0 || rows == 0) return ZDMMV_OK;
    if (!tma_shape_ok(fmt, cols)) return ZDMMV_ERR_SHAPE;  // the pipelined widths (multiples of 256, <= 8192)
    if (!w_stack || !idx || !x || !y) return ZDMMV_ERR_NULL;
    if (!aligned(w_stack, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(idx, 4) ||
        (status_dev && !aligned(status_dev, 4)))
        return ZDMMV_ERR_ALIGN;
    const int64_t nb = cols / kQK;
    const int64_t mat_bytes = rows * nb * block_bytes(fmt);
    if (expert_stride_bytes < 0 || x_stride < 0) return ZDMMV_ERR_SHAPE;
    if (n_experts > 1 && expert_stride_bytes < mat_bytes) return ZDMMV_ERR_SHAPE;
    if (x_stride != 0 && x_stride < cols) return ZDMMV_ERR_SHAPE;
    if (expert_stride_bytes % 16 || x_stride % 4) return ZDMMV_ERR_ALIGN;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w_stack);
    a.expert_stride = expert_stride_bytes;
    a.idx = idx;
    a.n_experts = n_experts;
    a.status = status_dev;
    a.xf = x;
    a.xf_stride = x_stride;
    a.y = y;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(nb);
    a.batch = 1;
    a.idx_ready = idx_ready ? 1 : 0;
    return run_dmmv(fmt, layout, a, n, st, true);
}

zdmmv_status argmax_entry(int fmt, const void *w, int layout, int64_t rows, int64_t cols, const void *xq,
                          int32_t *argmax_out, float *max_out, void *workspace, size_t workspace_bytes,
                          cudaStream_t st) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    if (rows <= 0 || rows > 0x7fffffff || !tma_shape_ok(fmt, cols)) return ZDMMV_ERR_SHAPE;
    if (!w || !xq || !argmax_out || !workspace) return ZDMMV_ERR_NULL;
    if (!aligned(w, 16) || !aligned(xq, 16) || !aligned(workspace, 16) || !aligned(argmax_out, 4) ||
        (max_out && !aligned(max_out, 4)))
        return ZDMMV_ERR_ALIGN;
    if (workspace_bytes < ZDMMV_ARGMAX_WORKSPACE_BYTES) return ZDMMV_ERR_SIZE;
    return from_cuda(launch_argmax_dmmv(fmt, layout, w, rows, cols, xq, argmax_out, max_out,
                                        static_cast<uint2 *>(workspace), st));
}

}  // namespace

cudaError_t launch_argmax_reduce(const uint2 *parts, int n, int32_t *argmax_out, float *max_out, cudaStream_t st,
                                 bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, argmax_reduce_kernel, parts, n, argmax_out, max_out);
}

cudaError_t launch_argmax_dmmv(int fmt, int layout, const void *w, int64_t rows, int64_t cols, const void *xq,
                               int32_t *argmax_out, float *max_out, uint2 *parts, cudaStream_t st) {
    const DeviceInfo *dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.rows = rows;
    a.nb = static_cast<int32_t>(cols / kQK);
    a.batch = 1;
    a.fault = dev->fault;
    a.argmax_parts = parts;
    const TmaPlan p = tma_plan(fmt, layout, cols, 1, kTmaWholeUnitMaxBytes);
    a.tile_rows = p.tile_rows;
    a.stage_bytes = p.stage_bytes;
    a.x_bytes_padded = p.x_bytes_padded;
    int per_sm = fmt == kFmtQ8 ? tma_ctas_per_sm_q8(layout, p) : tma_ctas_per_sm_q4(layout, p);
    const int want = ctas_per_sm_per_launch(rows * a.nb * static_cast<int64_t>(block_bytes(fmt)));
    if (per_sm > want) per_sm = want;
    int64_t ctas = static_cast<int64_t>(dev->sms) * per_sm;
    if (ctas > rows) ctas = rows;
    if (ctas > kArgmaxMaxCtas) ctas = kArgmaxMaxCtas;  // never more partials than `parts` holds
    e = fmt == kFmtQ8 ? launch_argmax_q8(a, p, layout, static_cast<int>(ctas), st, pdl_enabled())
                      : launch_argmax_q4(a, p, layout, static_cast<int>(ctas), st, pdl_enabled());
    if (e != cudaSuccess) return e;
    return launch_argmax_reduce(parts, static_cast<int>(ctas), argmax_out, max_out, st, pdl_enabled());
}

uint32_t *current_fault_word() {
    const DeviceInfo *dev = nullptr;
    return device_info(&dev) == cudaSuccess ? dev->fault : nullptr;
}

namespace {

zdmmv_status acc_entry(int fmt, const void *w, int layout, int64_t rows, int64_t cols, const void *xq,
                       const float *gate, float *y, cudaStream_t st) {
    zdmmv_status s = check_matrix(fmt, w, layout, rows, cols, xq, y);
    if (s != ZDMMV_OK) return s;
    if (rows == 0) return ZDMMV_OK;
    if (gate && !aligned(gate, 4)) return ZDMMV_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.y = y;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(cols / kQK);
    a.batch = 1;
    a.gate = gate;
    a.accumulate = 1;
    a.fault = dev->fault;
    if (!tma_shape_ok(fmt, cols)) return from_cuda(launch_plain(fmt, layout, a, 1, st));
    const TmaPlan p = tma_plan(fmt, layout, cols, 1, kTmaWholeUnitMaxBytes);
    a.tile_rows = p.tile_rows;
    a.stage_bytes = p.stage_bytes;
    a.x_bytes_padded = p.x_bytes_padded;
    int per_sm = fmt == kFmtQ8 ? tma_ctas_per_sm_q8(layout, p) : tma_ctas_per_sm_q4(layout, p);
    const int want = ctas_per_sm_per_launch(rows * a.nb * static_cast<int64_t>(block_bytes(fmt)));
    if (per_sm > want) per_sm = want;
    int64_t ctas = static_cast<int64_t>(dev->sms) * per_sm;
    if (ctas > rows) ctas = rows;
    if (ctas > 65535) ctas = 65535;
    return from_cuda(fmt == kFmtQ8 ? launch_acc_q8(a, p, layout, static_cast<int>(ctas), st, pdl_enabled())
                                   : launch_acc_q4(a, p, layout, static_cast<int>(ctas), st, pdl_enabled()));
}

zdmmv_status swiglu_entry(int fmt, const void *w_gate, const void *w_up, int64_t expert_stride_bytes, int layout,
                          int64_t rows, int64_t cols, const int32_t *idx, int n, int n_experts, const void *xq,
                          int64_t xq_stride_bytes, float *h, int32_t *status_dev, cudaStream_t st) {
    zdmmv_status s = check_matrix(fmt, w_gate, layout, rows, cols, xq, h);
    if (s != ZDMMV_OK) return s;
    if (!tma_shape_ok(fmt, cols)) return ZDMMV_ERR_SHAPE;
    if (n < 0 || n > 65535 || (!idx && n > 1) || n_experts < 0) return ZDMMV_ERR_SHAPE;
    if (n == 0 || rows == 0) return ZDMMV_OK;
    if (!w_up) return ZDMMV_ERR_NULL;
    if (!aligned(w_up, 16) || (idx && !aligned(idx, 4)) || (status_dev && !aligned(status_dev, 4)))
        return ZDMMV_ERR_ALIGN;
    const int64_t nb = cols / kQK;
    const int64_t mat_bytes = rows * nb * block_bytes(fmt);
    if (expert_stride_bytes < 0 || xq_stride_bytes < 0) return ZDMMV_ERR_SHAPE;
    if (idx && n_experts > 1 && expert_stride_bytes < mat_bytes) return ZDMMV_ERR_SHAPE;
    if (xq_stride_bytes != 0 && xq_stride_bytes < nb * 34) return ZDMMV_ERR_SHAPE;
    if (expert_stride_bytes % 16 || xq_stride_bytes % 16) return ZDMMV_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w_gate);
    a.w_b = static_cast<const uint8_t *>(w_up);
    a.slots_a = n;
    a.expert_stride = idx ? expert_stride_bytes : 0;
    a.idx = idx;
    a.n_experts = n_experts;
    a.status = status_dev;
    a.xq = static_cast<const uint8_t *>(xq);
    a.xq_stride = xq_stride_bytes;
    a.y = h;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(nb);
    a.batch = 1;
    a.fault = dev->fault;
    const TmaPlan p = tma_plan(fmt, layout, cols, 2);
    a.tile_rows = p.tile_rows;
    a.stage_bytes = p.stage_bytes;
    a.x_bytes_padded = p.x_bytes_padded;
    int per_sm = fmt == kFmtQ8 ? swiglu_ctas_per_sm_q8(layout, p) : swiglu_ctas_per_sm_q4(layout, p);
    const int want = ctas_per_sm_per_launch(2 * mat_bytes * n, a.idx != nullptr);
    if (per_sm > want) per_sm = want;
    int64_t ctas = static_cast<int64_t>(dev->sms) * per_sm / n;
    if (ctas < 1) ctas = 1;
    if (ctas > rows) ctas = rows;
    if (ctas > 65535) ctas = 65535;
    return from_cuda(fmt == kFmtQ8
                         ? launch_swiglu_q8(a, p, layout, static_cast<int>(ctas), n, st, pdl_enabled())
                         : launch_swiglu_q4(a, p, layout, static_cast<int>(ctas), n, st, pdl_enabled()));
}

zdmmv_status dmmv_xf32_entry(int fmt, const void *w, int layout, int64_t rows, int64_t cols, const float *x,
                             int batch, float *y, cudaStream_t st) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    if (rows < 0 || cols <= 0 || cols % kQK || cols / kQK > 0x3fffffff) return ZDMMV_ERR_SHAPE;
    if (batch < 1 || batch > ZDMMV_MAX_BATCH) return ZDMMV_ERR_SHAPE;
    if (rows == 0) return ZDMMV_OK;
    if (!w || !x || !y) return ZDMMV_ERR_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4)) return ZDMMV_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xf = x;
    a.xf_stride = cols;
    a.y = y;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(cols / kQK);
    a.batch = 1;
    a.fault = dev->fault;
    Xf32MmaPlan mp{};
    if (xf32_mma_plan(fmt, layout, rows, cols, &mp)) {
        // the fp16 tensor cores, the activation split into exact fp16 parts
        Xf32MmaArgs m{};
        m.w = a.w;
        m.xf = x;
        m.y = y;
        m.fault = dev->fault;
        m.rows = rows;
        m.xf_stride = cols;
        m.y_stride = rows;
        m.nb = a.nb;
        m.cb = mp.cb;
        m.nchunks = mp.nchunks;
        m.pitch = mp.pitch;
        return from_cuda(launch_xf32_mma(fmt, m, mp, batch, st, pdl_enabled()));
    }
    TmaPlan p{};
    if (xf32_plan(fmt, layout, cols, &p)) {
        a.tile_rows = p.tile_rows;
        a.stage_bytes = p.stage_bytes;
        a.x_bytes_padded = p.x_bytes_padded;
        // CTAs per slot: one wave of what fits (the launcher queries the occupancy)
        return from_cuda(fmt == kFmtQ8 ? launch_xf32_q8(a, p, layout, 0, batch, st, pdl_enabled())
                                       : launch_xf32_q4(a, p, layout, 0, batch, st, pdl_enabled()));
    }
    return from_cuda(fmt == kFmtQ8 ? launch_xf32_plain_q8(a, layout, dev->sms, batch, st, pdl_enabled())
                                   : launch_xf32_plain_q4(a, layout, dev->sms, batch, st, pdl_enabled()));
}

zdmmv_status dmmv_f32_entry(int fmt, const void *w, int layout, int64_t rows, int64_t cols, const float *x,
                            int batch, float *y, cudaStream_t st) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    if (rows < 0 || cols <= 0 || cols % kQK || cols / kQK > 0x3fffffff) return ZDMMV_ERR_SHAPE;
    if (batch < 1 || batch > ZDMMV_MAX_BATCH) return ZDMMV_ERR_SHAPE;
    if (rows == 0) return ZDMMV_OK;
    if (!w || !x || !y) return ZDMMV_ERR_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4)) return ZDMMV_ERR_ALIGN;
    DmmvArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xf = x;
    a.xf_stride = cols;
    a.y = y;
    a.y_stride = rows;
    a.rows = rows;
    a.nb = static_cast<int32_t>(cols / kQK);
    TmaPlan vp{};
    int vv = 0, nvg = 0;
    const int choice = batch_slots_forced() ? kBatchSlots : batch_kernel_choice();
    BmmaPlan hp{};
    if (batch >= 2 && (choice == kBatchMma || (choice == kBatchAuto && batch >= kBmmaMinBatch)) &&
        bmma_plan(fmt, layout, rows, cols, batch, &hp)) {
        // the batched call's tensor-core kernel with the quantization in its
        // prologue: the bits of the quantizer followed by zdmmv_q{8,4}_0_batched
        const DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
        if (choice == kBatchMma || (rows + kBmGroupRows - 1) / kBmGroupRows >= dev->sms) {
            BmmaArgs m{};
            m.w = a.w;
            m.xf = x;
            m.y = y;
            m.fault = dev->fault;
            m.rows = rows;
            m.y_stride = rows;
            m.nb = a.nb;
            m.batch = batch;
            m.nchunks = hp.nchunks;
            m.pitch = hp.pitch;
            m.red_bufs = hp.red_bufs;
            return from_cuda(launch_bmma(fmt, m, hp, true, st, pdl_enabled()));
        }
    }
    if (batch >= 2 && (choice == kBatchAuto || choice == kBatchVsplit) &&
        vsplit_plan(fmt, layout, cols, batch, &vp, &vv, &nvg)) {
        // one weight stream for the batch, its activations quantized in the prologue
        const DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
        a.fault = dev->fault;
        a.batch = batch;
        a.tile_rows = vp.tile_rows;
        a.stage_bytes = vp.stage_bytes;
        a.x_bytes_padded = vp.x_bytes_padded;
        const int cap = std::getenv("ZDMMV_BATCH_CTAS_PER_SM") ? batch_ctas_per_sm() : 0;
        cudaError_t e = fmt == kFmtQ8 ? launch_vsplit_fx_q8(a, vp, layout, vv, nvg, cap, st, pdl_enabled())
                                      : launch_vsplit_fx_q4(a, vp, layout, vv, nvg, cap, st, pdl_enabled());
        return from_cuda(e);
    }
    if (tma_shape_ok(fmt, cols)) {
        // single vectors, or batches the vector split does not take: one
        // fused single-vector launch with a slot per vector
        a.batch = 1;
        return run_dmmv(fmt, layout, a, batch, st, true);
    }
    if (static_cast<int64_t>(batch) * a.nb * 34 > kPlainFxMaxSmem) return ZDMMV_ERR_SHAPE;
    a.batch = batch;
    return run_dmmv(fmt, layout, a, 1, st, true);
}

}  // namespace
}  // namespace zdmmv

using namespace zdmmv;

// =================================================================== C ABI
extern "C" {

const char *zdmmv_status_str(zdmmv_status st) {
    switch (st) {
    case ZDMMV_OK: return "ok";
    case ZDMMV_ERR_NULL: return "null pointer";
    case ZDMMV_ERR_SHAPE: return "bad shape";
    case ZDMMV_ERR_ALIGN: return "misaligned pointer or stride";
    case ZDMMV_ERR_LAYOUT: return "unknown layout";
    case ZDMMV_ERR_FORMAT: return "unknown block format";
    case ZDMMV_ERR_SIZE: return "buffer too small";
    case ZDMMV_ERR_CUDA: return "CUDA runtime error";
    case ZDMMV_ERR_DEVICE: return "device fault reported";
    }
    return "unknown status";
}

const char *zdmmv_version(void) { return "zdmmv 0.1 (sm_103a)"; }

size_t zdmmv_block_bytes(zdmmv_fmt fmt) { return static_cast<size_t>(block_bytes(fmt)); }

zdmmv_status zdmmv_quantize_act_q8_0(const float *x, int64_t k, void *xq, zdmmv_stream_t stream) {
    if (k < 0 || k % kQK) return ZDMMV_ERR_SHAPE;
    if (k == 0) return ZDMMV_OK;
    if (!x || !xq) return ZDMMV_ERR_NULL;
    if (!aligned(x, 4)) return ZDMMV_ERR_ALIGN;
    const int64_t nblocks = k / kQK;
    const int64_t ctas = (nblocks + 7) / 8;
    if (ctas > 0x7fffffff) return ZDMMV_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return from_cuda(cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel, x, nblocks, static_cast<uint8_t *>(xq)));
}

zdmmv_status zdmmv_q8_0(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols, const void *xq, float *y,
                        zdmmv_stream_t stream) {
    return dmmv_entry(kFmtQ8, w, layout, rows, cols, xq, 1, y, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_q4_0(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols, const void *xq, float *y,
                        zdmmv_stream_t stream) {
    return dmmv_entry(kFmtQ4, w, layout, rows, cols, xq, 1, y, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_q8_0_batched(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols, const void *xq,
                                int batch, float *y, zdmmv_stream_t stream) {
    return dmmv_entry(kFmtQ8, w, layout, rows, cols, xq, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_q4_0_batched(const void *w, zdmmv_layout layout, int64_t rows, int64_t cols, const void *xq,
                                int batch, float *y, zdmmv_stream_t stream) {
    return dmmv_entry(kFmtQ4, w, layout, rows, cols, xq, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_expert_gather(zdmmv_fmt fmt, const void *w_stack, int64_t expert_stride_bytes,
                                 zdmmv_layout layout, int64_t rows, int64_t cols, const int32_t *idx, int n,
                                 int n_experts, const void *xq, int64_t xq_stride_bytes, float *y,
                                 int32_t *status_dev, zdmmv_stream_t stream) {
    return gather_entry(fmt, w_stack, nullptr, expert_stride_bytes, layout, rows, cols, idx, n, n_experts, xq,
                        xq_stride_bytes, y, nullptr, status_dev, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_expert_gather_ready(zdmmv_fmt fmt, const void *w_stack, int64_t expert_stride_bytes,
                                       zdmmv_layout layout, int64_t rows, int64_t cols, const int32_t *idx, int n,
                                       int n_experts, const void *xq, int64_t xq_stride_bytes, float *y,
                                       int32_t *status_dev, zdmmv_stream_t stream) {
    return gather_entry(fmt, w_stack, nullptr, expert_stride_bytes, layout, rows, cols, idx, n, n_experts, xq,
                        xq_stride_bytes, y, nullptr, status_dev, reinterpret_cast<cudaStream_t>(stream), true);
}

zdmmv_status zdmmv_expert_gather_f32(zdmmv_fmt fmt, const void *w_stack, int64_t expert_stride_bytes,
                                     zdmmv_layout layout, int64_t rows, int64_t cols, const int32_t *idx, int n,
                                     int n_experts, const float *x, int64_t x_stride, float *y,
                                     int32_t *status_dev, int idx_ready, zdmmv_stream_t stream) {
    return gather_f32_entry(fmt, w_stack, expert_stride_bytes, layout, rows, cols, idx, n, n_experts, x, x_stride,
                            y, status_dev, idx_ready != 0, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_expert_gather2(zdmmv_fmt fmt, const void *w_stack_a, const void *w_stack_b,
                                  int64_t expert_stride_bytes, zdmmv_layout layout, int64_t rows, int64_t cols,
                                  const int32_t *idx, int n, int n_experts, const void *xq,
                                  int64_t xq_stride_bytes, float *y_a, float *y_b, int32_t *status_dev,
                                  zdmmv_stream_t stream) {
    if (!w_stack_b || !y_b) return n == 0 || rows == 0 ? ZDMMV_OK : ZDMMV_ERR_NULL;
    return gather_entry(fmt, w_stack_a, w_stack_b, expert_stride_bytes, layout, rows, cols, idx, n, n_experts, xq,
                        xq_stride_bytes, y_a, y_b, status_dev, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_dmmv_f32(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                            const float *x, int batch, float *y, zdmmv_stream_t stream) {
    return dmmv_f32_entry(fmt, w, layout, rows, cols, x, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_dmmv_argmax(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                               const void *xq, int32_t *argmax_out, float *max_out, void *workspace,
                               size_t workspace_bytes, zdmmv_stream_t stream) {
    return argmax_entry(fmt, w, layout, rows, cols, xq, argmax_out, max_out, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_dmmv_xf32(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                             const float *x, int batch, float *y, zdmmv_stream_t stream) {
    return dmmv_xf32_entry(fmt, w, layout, rows, cols, x, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

size_t zdmmv_expert_ffn_workspace_bytes(int n, int64_t ffn) { return ffn_workspace_bytes(n, ffn); }

zdmmv_status zdmmv_expert_ffn(zdmmv_fmt fmt_gate_up, const void *w_gate, const void *w_up,
                              int64_t gate_up_stride_bytes, zdmmv_fmt fmt_down, const void *w_down,
                              int64_t down_stride_bytes, int64_t hidden, int64_t ffn, const int32_t *idx, int n,
                              int n_experts, const void *xq, float *y, void *workspace, size_t workspace_bytes,
                              int32_t *status_dev, zdmmv_stream_t stream) {
    return static_cast<zdmmv_status>(ffn_entry_status(fmt_gate_up, w_gate, w_up, gate_up_stride_bytes, fmt_down,
                                                      w_down, down_stride_bytes, hidden, ffn, idx, n, n_experts, xq,
                                                      y, workspace, workspace_bytes, status_dev,
                                                      reinterpret_cast<cudaStream_t>(stream), pdl_enabled()));
}

zdmmv_status zdmmv_expert_swiglu(zdmmv_fmt fmt, const void *w_gate, const void *w_up, int64_t expert_stride_bytes,
                                 zdmmv_layout layout, int64_t rows, int64_t cols, const int32_t *idx, int n,
                                 int n_experts, const void *xq, int64_t xq_stride_bytes, float *h,
                                 int32_t *status_dev, zdmmv_stream_t stream) {
    return swiglu_entry(fmt, w_gate, w_up, expert_stride_bytes, layout, rows, cols, idx, n, n_experts, xq,
                        xq_stride_bytes, h, status_dev, reinterpret_cast<cudaStream_t>(stream));
}

zdmmv_status zdmmv_dmmv_acc(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                            const void *xq, const float *gate, float *y, zdmmv_stream_t stream) {
    return acc_entry(fmt, w, layout, rows, cols, xq, gate, y, reinterpret_cast<cudaStream_t>(stream));
}

size_t zdmmv_repacked_bytes(zdmmv_fmt fmt, int64_t rows, int64_t cols) {
    if (block_bytes(fmt) == 0 || rows < 0 || cols <= 0 || cols % kQK) return 0;
    return static_cast<size_t>(rows * (cols / kQK) * block_bytes(fmt));
}

zdmmv_status zdmmv_repack(zdmmv_fmt fmt, const void *src, int64_t rows, int64_t cols, void *dst, size_t dst_bytes,
                          zdmmv_stream_t stream) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (rows < 0 || cols <= 0 || cols % kQK) return ZDMMV_ERR_SHAPE;
    if (rows == 0) return ZDMMV_OK;
    if (!src || !dst) return ZDMMV_ERR_NULL;
    if (!aligned(src, 16) || !aligned(dst, 16)) return ZDMMV_ERR_ALIGN;
    const size_t need = zdmmv_repacked_bytes(fmt, rows, cols);
    if (dst_bytes < need) return ZDMMV_ERR_SIZE;
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    if (s8 < d8 + need && d8 < s8 + need) return ZDMMV_ERR_SHAPE;  // overlapping buffers
    const int64_t nblocks = rows * (cols / kQK);
    const int64_t ctas = (nblocks + 255) / 256;
    if (ctas > 0x7fffffff) return ZDMMV_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(fmt == ZDMMV_Q8_0 ? launch_plain_cfg(repack_kernel<kFmtQ8>, static_cast<unsigned>(ctas), 256, st,
                                                          s8, nblocks, d8)
                                       : launch_plain_cfg(repack_kernel<kFmtQ4>, static_cast<unsigned>(ctas), 256, st,
                                                          s8, nblocks, d8));
}

size_t zdmmv_host_step_workspace_bytes(int64_t rows, int64_t cols, int batch) {
    if (rows < 0 || cols <= 0 || cols % kQK || batch < 1 || batch > ZDMMV_MAX_BATCH) return 0;
    const int64_t xb = round_up(static_cast<int64_t>(batch) * cols * 4, 256);
    const int64_t qb = round_up(static_cast<int64_t>(batch) * (cols / kQK) * 34, 256);
    const int64_t yb = round_up(static_cast<int64_t>(batch) * rows * 4, 256);
    return static_cast<size_t>(xb + qb + yb);
}

namespace {
// The device address of a host buffer of `bytes` bytes when the whole buffer is
// page-locked memory of ONE allocation mapped into the current context (a
// kernel may then read or write it directly, over the chip-to-chip link on a
// Grace system), else nullptr: both ends are looked up and must be host memory
// of the same allocation (buffer id) at linear device addresses.
void *mapped_host_buffer(const void *p, size_t bytes) {
    static const PFN_cuPointerGetAttributes_v7000 get = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuPointerGetAttributes_v7000>(nullptr);
        return reinterpret_cast<PFN_cuPointerGetAttributes_v7000>(f);
    }();
    if (!get || !p || bytes == 0) return nullptr;
    struct End {
        unsigned int type = 0;
        CUdeviceptr dptr = 0;
        unsigned long long id = 0;
    } e[2];
    const uintptr_t a[2] = {reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + bytes - 1};
    for (int i = 0; i < 2; ++i) {
        CUpointer_attribute at[3] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_POINTER,
                                     CU_POINTER_ATTRIBUTE_BUFFER_ID};
        void *data[3] = {&e[i].type, &e[i].dptr, &e[i].id};
        // an address CUDA does not know yields zeros, not an error
        if (get(3, at, data, static_cast<CUdeviceptr>(a[i])) != CUDA_SUCCESS) return nullptr;
        if (e[i].type != CU_MEMORYTYPE_HOST || e[i].dptr == 0 || e[i].id == 0) return nullptr;
    }
    if (e[0].id != e[1].id || e[1].dptr - e[0].dptr != bytes - 1) return nullptr;
    return reinterpret_cast<void *>(e[0].dptr);
}
}  // namespace

zdmmv_status zdmmv_host_step(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                             const float *x_host, int batch, float *y_host, void *workspace_dev,
                             size_t workspace_bytes, zdmmv_stream_t stream) {
    if (block_bytes(fmt) == 0) return ZDMMV_ERR_FORMAT;
    if (rows < 0 || cols <= 0 || cols % kQK || batch < 1 || batch > ZDMMV_MAX_BATCH) return ZDMMV_ERR_SHAPE;
    if (!w || !x_host || !y_host || !workspace_dev) return ZDMMV_ERR_NULL;
    if (!aligned(workspace_dev, 16)) return ZDMMV_ERR_ALIGN;
    if (workspace_bytes < zdmmv_host_step_workspace_bytes(rows, cols, batch)) return ZDMMV_ERR_SIZE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace_dev);
    const int64_t xb = round_up(static_cast<int64_t>(batch) * cols * 4, 256);
    const int64_t qb = round_up(static_cast<int64_t>(batch) * (cols / kQK) * 34, 256);
    float *xd = reinterpret_cast<float *>(ws);
    uint8_t *xqd = ws + xb;
    float *yd = reinterpret_cast<float *>(ws + xb + qb);
    const size_t x_bytes = static_cast<size_t>(batch) * cols * 4;
    const size_t y_bytes = static_cast<size_t>(batch) * rows * 4;
    if (rows > 0) {
        // page-locked host buffers: no copies; the quantizer reads x from host
        // memory once and the DMMV stores y into host memory (the same bits as
        // the fused launch)
        const float *xm = static_cast<const float *>(mapped_host_buffer(x_host, x_bytes));
        float *ym = static_cast<float *>(mapped_host_buffer(y_host, y_bytes));
        if (xm && ym && aligned(ym, 4)) {
            zdmmv_status s = zdmmv_quantize_act_q8_0(xm, static_cast<int64_t>(batch) * cols, xqd, stream);
            if (s != ZDMMV_OK) return s;
            return dmmv_entry(fmt, w, layout, rows, cols, xqd, batch, ym, st);
        }
    }
    cudaError_t e = cudaMemcpyAsync(xd, x_host, x_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return ZDMMV_ERR_CUDA;
    zdmmv_status s;
    if (tma_shape_ok(fmt, cols) && batch == 1) {
        // quantize + DMMV in one launch: the same bits as the quantizer followed by the DMMV
        s = dmmv_f32_entry(fmt, w, layout, rows, cols, xd, batch, yd, st);
    } else {
        s = zdmmv_quantize_act_q8_0(xd, static_cast<int64_t>(batch) * cols, xqd, stream);
        if (s == ZDMMV_OK) s = dmmv_entry(fmt, w, layout, rows, cols, xqd, batch, yd, st);
    }
    if (s != ZDMMV_OK) return s;
    if (rows > 0) {
        e = cudaMemcpyAsync(y_host, yd, y_bytes, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return ZDMMV_ERR_CUDA;
    }
    return ZDMMV_OK;
}

zdmmv_status zdmmv_debug_block_sums(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows, int64_t cols,
                                    const void *xq, int32_t *sums, zdmmv_stream_t stream) {
    zdmmv_status s = check_matrix(fmt, w, layout, rows, cols, xq, reinterpret_cast<const float *>(sums));
    if (s != ZDMMV_OK) return s;
    if (rows == 0) return ZDMMV_OK;
    const int nb = static_cast<int>(cols / kQK);
    const bool pairs = tma_shape_ok(fmt, cols);
    const int64_t threads = pairs ? rows * (nb / 2) : rows * nb;
    const int64_t ctas = (threads + 255) / 256;
    if (ctas > 0x7fffffff) return ZDMMV_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *w8 = static_cast<const uint8_t *>(w);
    const uint8_t *x8 = static_cast<const uint8_t *>(xq);
    const unsigned g = static_cast<unsigned>(ctas);
    cudaError_t e = cudaSuccess;
#define ZDMMV_SUMS(F, L, PR) e = launch_plain_cfg(block_sums_kernel<F, L, PR>, g, 256, st, w8, rows, nb, x8, sums)
    if (fmt == ZDMMV_Q8_0) {
        if (layout == ZDMMV_LAYOUT_GGUF) {
            if (pairs) ZDMMV_SUMS(kFmtQ8, kLayoutGguf, true); else ZDMMV_SUMS(kFmtQ8, kLayoutGguf, false);
        } else {
            if (pairs) ZDMMV_SUMS(kFmtQ8, kLayoutRepacked, true); else ZDMMV_SUMS(kFmtQ8, kLayoutRepacked, false);
        }
    } else {
        if (layout == ZDMMV_LAYOUT_GGUF) {
            if (pairs) ZDMMV_SUMS(kFmtQ4, kLayoutGguf, true); else ZDMMV_SUMS(kFmtQ4, kLayoutGguf, false);
        } else {
            if (pairs) ZDMMV_SUMS(kFmtQ4, kLayoutRepacked, true); else ZDMMV_SUMS(kFmtQ4, kLayoutRepacked, false);
        }
    }
#undef ZDMMV_SUMS
    return from_cuda(e);
}

zdmmv_status zdmmv_selftest_dp4a(const int32_t *a, const int32_t *b, const int32_t *c, int32_t *out, int n,
                                 zdmmv_stream_t stream) {
    if (n < 0) return ZDMMV_ERR_SHAPE;
    if (n == 0) return ZDMMV_OK;
    if (!a || !b || !c || !out) return ZDMMV_ERR_NULL;
    return from_cuda(launch_plain_cfg(selftest_dp4a_kernel, static_cast<unsigned>((n + 255) / 256), 256,
                                      reinterpret_cast<cudaStream_t>(stream), a, b, c, out, n));
}

zdmmv_status zdmmv_selftest_wait_timeout(int32_t *result, zdmmv_stream_t stream) {
    if (!result) return ZDMMV_ERR_NULL;
    const DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return ZDMMV_ERR_CUDA;
    return from_cuda(launch_plain_cfg(selftest_wait_timeout_kernel, 1, 32, reinterpret_cast<cudaStream_t>(stream),
                                      dev->fault, result));
}

zdmmv_status zdmmv_device_status(uint32_t *bits_out, int clear) {
    if (!bits_out) return ZDMMV_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return ZDMMV_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v)) != cudaSuccess) return ZDMMV_ERR_CUDA;
    if (clear) {
        const uint32_t z = 0;
        if (cudaMemcpyToSymbol(g_fault_word, &z, sizeof(z)) != cudaSuccess) return ZDMMV_ERR_CUDA;
    }
    *bits_out = v;
    return ZDMMV_OK;
}

}  // extern "C"
