// zdmmv_xf32.cuh -- the decode DMMV with the activation taken as fp32 values
// (no Q8_0 quantization of x), for sm_103a.
//
// y[r] = sum_b d_w * sum_i v_i * x_i: each weight block is dequantized in
// registers and multiplied by the fp32 input vector, as the ZINC_RT Q8_0 slice
// does with its f32 input ("The first ZINC_RT model slices that actually
// count", kernel ABI) and as the Vulkan DMMV does with x staged in shared memory
// (habr ZINC article, "Что такое DMMV", "Трюк с shared memory").
//
// Weights stream through the same TMA ring as the quantized kernel (producer
// warp, full/empty mbarriers, weight tiles prefetched before the dependency
// wait). The activation is copied once per CTA into shared memory with a 16-byte
// pad after every 32-value block, so the 8 lanes of a 128-bit load phase that
// read 8 consecutive blocks hit 8 different bank groups.
//
// Lane l of a row group (LPR lanes) owns blocks l, l+LPR, ...; for each owned
// block it loads the block's 32 x values once and applies them to R rows. A
// weight value becomes an exact float without a conversion instruction: its byte
// (offset to 0..255, or the 4-bit code 0..15) is placed in the low mantissa bits
// of 2^23 by one byte permute, and one add removes 2^23 plus the offset. Four
// fp32 fma chains per block and row, combined in a fixed order, then
// acc = fma(d_w, block_sum, acc); the row's lanes meet in an xor-shuffle tree.
#pragma once

#include "zdmmv_batch.cuh"

namespace zdmmv {

constexpr int kXf32BlockStride = 144;  // shared-memory bytes per activation block (128 + 16 pad)

__device__ __forceinline__ void sts128(uint32_t a, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Byte C of w as the float 2^23 + byte, minus bias (exact for bytes 0..255).
template <int C>
__device__ __forceinline__ float byte_value(uint32_t w, float bias) {
    return __fadd_rn(__int_as_float(static_cast<int>(__byte_perm(w, 0x4B000000u, 0x7540u + C))), -bias);
}

// sum_i v_i * x_i over one block, in four chains combined as (c0 + c1) + (c2 + c3).
// q: the block's aligned quant words; x: its 32 activation values.
template <int FMT> struct XfBlock;

template <> struct XfBlock<kFmtQ8> {
    // chain c takes words c and c + 4 (elements 4c..4c+3 and 16+4c..16+4c+3)
    __device__ __forceinline__ static float dot(const uint32_t (&q)[8], const float (&x)[32]) {
        constexpr float kBias = 8388608.0f + 128.0f;
        float c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a = q[k] ^ 0x80808080u;  // int8 -> offset binary
            const uint32_t b = q[k + 4] ^ 0x80808080u;
            float t = __fmul_rn(byte_value<0>(a, kBias), x[4 * k]);
            t = __fmaf_rn(byte_value<1>(a, kBias), x[4 * k + 1], t);
            t = __fmaf_rn(byte_value<2>(a, kBias), x[4 * k + 2], t);
            t = __fmaf_rn(byte_value<3>(a, kBias), x[4 * k + 3], t);
            t = __fmaf_rn(byte_value<0>(b, kBias), x[16 + 4 * k], t);
            t = __fmaf_rn(byte_value<1>(b, kBias), x[16 + 4 * k + 1], t);
            t = __fmaf_rn(byte_value<2>(b, kBias), x[16 + 4 * k + 2], t);
            t = __fmaf_rn(byte_value<3>(b, kBias), x[16 + 4 * k + 3], t);
            c[k] = t;
        }
        return __fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3]));
    }
};

template <> struct XfBlock<kFmtQ4> {
    // chain k takes qs word k: low nibbles = elements 4k..4k+3, high = 16+4k..16+4k+3
    __device__ __forceinline__ static float dot(const uint32_t (&q)[4], const float (&x)[32]) {
        constexpr float kBias = 8388608.0f + 8.0f;
        float c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = q[k] & kLoNib;
            const uint32_t hi = (q[k] >> 4) & kLoNib;
            float t = __fmul_rn(byte_value<0>(lo, kBias), x[4 * k]);
            t = __fmaf_rn(byte_value<1>(lo, kBias), x[4 * k + 1], t);
            t = __fmaf_rn(byte_value<2>(lo, kBias), x[4 * k + 2], t);
            t = __fmaf_rn(byte_value<3>(lo, kBias), x[4 * k + 3], t);
            t = __fmaf_rn(byte_value<0>(hi, kBias), x[16 + 4 * k], t);
            t = __fmaf_rn(byte_value<1>(hi, kBias), x[16 + 4 * k + 1], t);
            t = __fmaf_rn(byte_value<2>(hi, kBias), x[16 + 4 * k + 2], t);
            t = __fmaf_rn(byte_value<3>(hi, kBias), x[16 + 4 * k + 3], t);
            c[k] = t;
        }
        return __fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3]));
    }
};

// The 32 activation values of block b from the padded shared-memory copy.
__device__ __forceinline__ void load_x_f32(uint32_t xs, int b, float (&x)[32]) {
    const uint32_t base = xs + static_cast<uint32_t>(b * kXf32BlockStride);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 v = lds128(base + 16 * k);
        x[4 * k] = __uint_as_float(v.x);
        x[4 * k + 1] = __uint_as_float(v.y);
        x[4 * k + 2] = __uint_as_float(v.z);
        x[4 * k + 3] = __uint_as_float(v.w);
    }
}

// Pipelined kernel. a.xf / a.xf_stride: fp32 activation per slot (blockIdx.y);
// a.y / a.y_stride: output per slot. R rows per row group at a time.
template <int FMT, int LAYOUT, int LPR, int R, int STAGES>
__global__ void __launch_bounds__(kTmaThreads, 3) dmmv_xf32_kernel(const DmmvArgs a) {
    constexpr int kRowsPar = kConsumerThreads / LPR;
    constexpr int kQW = Fmt<FMT>::kQuantBytes / 4;
    static_assert(kConsumerThreads % LPR == 0 && LPR <= 32, "row groups live inside a warp");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xready = empty + STAGES;  // the consumers have staged the activation
    uint8_t *xs = smem + kBarrierBytes;
    uint8_t *stage0 = xs + a.x_bytes_padded;

    const int tid = threadIdx.x;
    const int slot = blockIdx.y;
    const int64_t rows = a.rows;
    const int64_t r0 = rows * blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (blockIdx.x + 1) / gridDim.x;
    const int nb = a.nb;
    float *y = a.y + slot * a.y_stride;
    const float *x = a.xf + slot * a.xf_stride;

    pdl_launch_dependents();
    if (r1 <= r0) return;
    const int T = a.tile_rows;
    const int ntiles = static_cast<int>((r1 - r0 + T - 1) / T);

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerThreads / 32);
        }
        mbar_init(xready, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        // ------------------------------------------------------- producer
        if (tid != kConsumerThreads) return;
        const uint64_t wpol = l2_evict_first_policy();
        // One tile streams before the consumers' activation loads, the rest of the
        // ring once the activation is staged: loads issued behind the whole ring
        // of this CTA's weight copies would wait for all of them.
        const int nring = ntiles < STAGES ? ntiles : STAGES;
        issue_tile<FMT, LAYOUT>(a, a.w, r0, r1, 0, 0, stage0, full, wpol);
        int issued = 1;
        bool ok = mbar_wait(xready, 0);
        for (; ok && issued < nring; ++issued) issue_tile<FMT, LAYOUT>(a, a.w, r0, r1, issued, issued, stage0, full, wpol);
        for (int t = issued; ok && t < ntiles; ++t) {
            const int s = t % STAGES;
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((t / STAGES) - 1) & 1u)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            issue_tile<FMT, LAYOUT>(a, a.w, r0, r1, t, s, stage0, full, wpol);
            issued = t + 1;
        }
        if (!ok) atomicOr(a.fault, 1u);
        for (int s = 0; s < STAGES; ++s) {
            const int t_last = (issued - 1 - s) >= 0 ? ((issued - 1 - s) / STAGES) * STAGES + s : -1;
            if (t_last >= 0) (void)mbar_wait(&full[s], static_cast<uint32_t>(t_last / STAGES) & 1u);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int g = tid / LPR;
    const int l = tid % LPR;
    const uint32_t xsa = smem_addr(xs);
    pdl_wait();  // the activation may be written, and y still read, by the preceding kernel
    {
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        const int nq = nb * 8;
        for (int q = tid; q < nq; q += kConsumerThreads)
            sts128(xsa + static_cast<uint32_t>((q >> 3) * kXf32BlockStride + (q & 7) * 16), x4[q]);
    }
    consumer_barrier();
    if (tid == 0) mbar_arrive(xready);
    const int bpl = nb / LPR;  // nb is a multiple of LPR on this path

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
        const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * a.stage_bytes);
        const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
        const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
        for (int base = 0; base < nr; base += kRowsPar * R) {
            float acc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r] = 0.0f;
            for (int j = 0; j < bpl; ++j) {
                const int b = l + j * LPR;
                float xv[32];
                load_x_f32(xsa, b, xv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int i = base + r * kRowsPar + g;
                    if (i < nr) {
                        uint32_t q[kQW];
                        float dw;
                        load_wblock<FMT, LAYOUT>(st, i, b, nb, T, q, dw);
                        acc[r] = __fmaf_rn(dw, XfBlock<FMT>::dot(q, xv), acc[r]);
                    }
                }
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int i = base + r * kRowsPar + g;
                if (l == 0 && i < nr) y[tr0 + i] = acc[r];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// Plain kernel for widths off the pipelined path (any multiple of 32 columns):
// one warp per row, lane l takes blocks l, l+32, ..., x read from global memory.
template <int FMT, int LAYOUT>
__global__ void __launch_bounds__(256) dmmv_xf32_plain_kernel(const DmmvArgs a) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int nb = a.nb;
    const int slot = blockIdx.y;
    const float *x = a.xf + slot * a.xf_stride;
    float *y = a.y + slot * a.y_stride;
    for (int64_t r = wid; r < a.rows; r += warps) {
        float acc = 0.0f;
        for (int b = lane; b < nb; b += 32) {
            float xv[32];
            const float4 *x4 = reinterpret_cast<const float4 *>(x + static_cast<int64_t>(b) * kQK);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = x4[k];
                xv[4 * k] = v.x;
                xv[4 * k + 1] = v.y;
                xv[4 * k + 2] = v.z;
                xv[4 * k + 3] = v.w;
            }
            uint32_t q8[8];
            float dw;
            if constexpr (LAYOUT == kLayoutGguf)
                Block<FMT>::load_gguf(a.w + (r * nb + b) * kBB, q8, dw);
            else
                Block<FMT>::load_repacked(a.w + (r * nb + b) * kQB, a.w + a.rows * nb * kQB + (r * nb + b) * 2, q8,
                                          dw);
            if constexpr (FMT == kFmtQ8) {
                acc = __fmaf_rn(dw, XfBlock<FMT>::dot(q8, xv), acc);
            } else {
                const uint32_t q4[4] = {q8[0], q8[1], q8[2], q8[3]};
                acc = __fmaf_rn(dw, XfBlock<FMT>::dot(q4, xv), acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) y[r] = acc;
    }
}

template <int FMT, int LAYOUT, int LPR, int R, int STAGES>
struct Xf32Inst {
    static constexpr auto kKernel = &dmmv_xf32_kernel<FMT, LAYOUT, LPR, R, STAGES>;
    // ctas_per_slot <= 0: one wave of the CTAs that fit on the device, split over the slots
    static cudaError_t launch(const DmmvArgs &a, const TmaPlan &p, int ctas_per_slot, int slots, cudaStream_t st,
                              bool pdl) {
        static std::atomic<bool> done[64];  // smem limit raised, per device
        static std::atomic<uint64_t> occ_cache[64];  // (smem << 32) | CTAs per SM, per device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!done[dev].load(std::memory_order_acquire)) {
            e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kKernel), dev);
            if (e != cudaSuccess) return e;
            done[dev].store(true, std::memory_order_release);
        }
        if (ctas_per_slot <= 0) {
            int per_sm = 0;
            const uint64_t c = occ_cache[dev].load(std::memory_order_relaxed);
            if (c != 0 && static_cast<int>(c >> 32) == p.smem_bytes) {
                per_sm = static_cast<int>(c & 0xffffffffu);
            } else {
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kKernel, kTmaThreads,
                                                                  static_cast<size_t>(p.smem_bytes));
                if (e != cudaSuccess) return e;
                per_sm = per_sm > 0 ? per_sm : 1;
                occ_cache[dev].store((static_cast<uint64_t>(p.smem_bytes) << 32) | static_cast<uint32_t>(per_sm),
                                     std::memory_order_relaxed);
            }
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            int64_t n = static_cast<int64_t>(sms) * per_sm / slots;
            if (n < 1) n = 1;
            if (n > a.rows) n = a.rows;
            ctas_per_slot = static_cast<int>(n);
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas_per_slot), static_cast<unsigned>(slots), 1);
        cfg.blockDim = dim3(kTmaThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kKernel, a);
    }
};

// p.lpr lanes per row, p.ppl = R rows per row group at a time, p.stages 2 or 3.
template <int FMT, int LAYOUT>
cudaError_t launch_xf32_layout(const DmmvArgs &a, const TmaPlan &p, int ctas_per_slot, int slots, cudaStream_t st,
                               bool pdl) {
#define ZDMMV_XVAR(LPR_, R_, ST_)                                          \
    if (p.lpr == LPR_ && p.ppl == R_ && p.stages == ST_)                   \
        return Xf32Inst<FMT, LAYOUT, LPR_, R_, ST_>::launch(a, p, ctas_per_slot, slots, st, pdl);
#define ZDMMV_XVAR_ST(LPR_, R_) ZDMMV_XVAR(LPR_, R_, 2) ZDMMV_XVAR(LPR_, R_, 3)
    ZDMMV_XVAR_ST(32, 4)
    ZDMMV_XVAR_ST(32, 2)
    ZDMMV_XVAR_ST(32, 1)
    ZDMMV_XVAR_ST(16, 4)
    ZDMMV_XVAR_ST(16, 2)
    ZDMMV_XVAR_ST(16, 1)
    ZDMMV_XVAR_ST(8, 4)
    ZDMMV_XVAR_ST(8, 2)
    ZDMMV_XVAR_ST(8, 1)
#undef ZDMMV_XVAR_ST
#undef ZDMMV_XVAR
    return cudaErrorInvalidConfiguration;
}

template <int FMT>
cudaError_t launch_xf32_fmt(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                            cudaStream_t st, bool pdl) {
    if (layout == kLayoutGguf) return launch_xf32_layout<FMT, kLayoutGguf>(a, p, ctas_per_slot, slots, st, pdl);
    return launch_xf32_layout<FMT, kLayoutRepacked>(a, p, ctas_per_slot, slots, st, pdl);
}

template <int FMT>
cudaError_t launch_xf32_plain_fmt(const DmmvArgs &a, int layout, int sms, int slots, cudaStream_t st, bool pdl) {
    int64_t ctas = (a.rows + 7) / 8;
    if (ctas > static_cast<int64_t>(sms) * 8) ctas = static_cast<int64_t>(sms) * 8;
    if (ctas < 1) ctas = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), static_cast<unsigned>(slots), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (layout == kLayoutGguf) return cudaLaunchKernelEx(&cfg, dmmv_xf32_plain_kernel<FMT, kLayoutGguf>, a);
    return cudaLaunchKernelEx(&cfg, dmmv_xf32_plain_kernel<FMT, kLayoutRepacked>, a);
}

}  // namespace zdmmv
