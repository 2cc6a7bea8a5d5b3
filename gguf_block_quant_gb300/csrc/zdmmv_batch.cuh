// zdmmv_batch.cuh -- batched decode DMMV: one weight stream, up to 8 activation
// vectors (sm_103a).
//
// The weight tiles are streamed exactly as in the single-vector kernel (bulk
// TMA into a shared-memory ring by a producer warp, prefetched before the
// dependency wait), but each tile is dotted against all B vectors before it is
// released, so HBM sees the weights once per call whatever B is.
//
// Work split (4 consumer warps, 128 threads): a row group of G threads covers one
// row; thread t of the group owns blocks t, t+G, ... of the row (BPT blocks). The
// codes of VB activation vectors for the owned blocks are held in registers
// (one "pass"); B > VB vectors take several passes over the same shared-memory
// tile, so shared memory, not HBM, absorbs the re-reads. Each group computes two
// rows at a time; the 2*VB partial sums of a warp are combined with a
// reduce-scatter (halving exchanges), then across the group's warps through
// shared memory.
//
// Block arithmetic is the same as everywhere else (dp4a per 4 bytes, Q4_0 nibble
// unpack with the -8 offset folded into the accumulator, fp32 fma with the exact
// d_w*d_x product). In the GGUF layout a block starts 0 or 2 bytes into a word
// (34 and 18 are 2 mod 4); the thread knows its block's parity and holds its
// activation words shifted to match, with zeros facing the fp16 scale bytes.
#pragma once

#include "zdmmv_tma.cuh"

namespace zdmmv {

// Registers for one owned block of one vector: its 32 codes as 8 aligned words
// (Q4_0: split into the codes facing the low and the high nibbles), the -8 offset
// term (Q4_0) and the fp16 scale as float.
template <int FMT> struct BVec;

template <> struct BVec<kFmtQ8> {
    uint32_t x[8];
    float dx;
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = 0;
        dx = 0.0f;
    }
    __device__ __forceinline__ void set(const uint32_t (&w)[8], float d) {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = w[k];
        dx = d;
    }
    // q: the block's 8 aligned quant words
    __device__ __forceinline__ int dot(const uint32_t (&q)[8]) const {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a_ss(q[k], x[k], s);
        return s;
    }
};

template <> struct BVec<kFmtQ4> {
    uint32_t xlo[4], xhi[4];
    int init;
    float dx;
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int k = 0; k < 4; ++k) xlo[k] = xhi[k] = 0;
        init = 0;
        dx = 0.0f;
    }
    __device__ __forceinline__ void set(const uint32_t (&xw)[8], float d) {
        dx = d;
        init = q4_offset_term(xw);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            xlo[k] = xw[k];
            xhi[k] = xw[4 + k];
        }
    }
    // lo / hi: the block's 4 aligned qs words masked to low nibbles / high nibbles (16*q)
    __device__ __forceinline__ int dot(const uint32_t (&lo)[4], const uint32_t (&hi)[4]) const {
        int l = init, h = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            l = dp4a_ss(lo[k], xlo[k], l);
            h = dp4a_us(hi[k], xhi[k], h);
        }
        return l + (h >> 4);
    }
};

// The aligned quant words (QW of them) and the scale of a block stored at byte
// offset `off` (even) from a 4-byte aligned base: the block starts 0 or 2 bytes
// into a word; for the latter the quant words need no realignment (w0 holds the
// scale in its high half), for the former each word is realigned with one byte
// permute. Works for shared or global memory.
template <int QW>
__device__ __forceinline__ void load_block_aligned(const uint8_t *base, int64_t off, uint32_t (&q)[QW], float &d) {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(base + (off & ~int64_t(3)));
    uint32_t w[QW + 1];
#pragma unroll
    for (int k = 0; k <= QW; ++k) w[k] = src[k];
    if (off & 2) {  // w0 = [.. .. d d], quants aligned in w1..
        d = half_hi(w[0]);
#pragma unroll
        for (int k = 0; k < QW; ++k) q[k] = w[k + 1];
    } else {        // w0 = [d d q0 q1], quants shifted by 2 bytes
        d = half_lo(w[0]);
#pragma unroll
        for (int k = 0; k < QW; ++k) q[k] = shift2(w[k], w[k + 1]);
    }
}

// The same from shared memory (base: shared-memory address, 4-byte aligned).
template <int QW>
__device__ __forceinline__ void load_block_aligned_smem(uint32_t base, int off, uint32_t (&q)[QW], float &d) {
    const uint32_t src = base + static_cast<uint32_t>(off & ~3);
    uint32_t w[QW + 1];
#pragma unroll
    for (int k = 0; k <= QW; ++k) w[k] = lds32(src + 4 * k);
    if (off & 2) {
        d = half_hi(w[0]);
#pragma unroll
        for (int k = 0; k < QW; ++k) q[k] = w[k + 1];
    } else {
        d = half_lo(w[0]);
#pragma unroll
        for (int k = 0; k < QW; ++k) q[k] = shift2(w[k], w[k + 1]);
    }
}

// The aligned quant words and scale of block b of staged row i. GGUF blocks start
// 0 (even b) or 2 (odd b) bytes into a word; for an even block the quant words are
// realigned once (one byte permute per word) and then serve every vector.
template <int FMT, int LAYOUT>
__device__ __forceinline__ void load_wblock(uint32_t stage, int i, int b, int nb, int tile_rows,
                                            uint32_t (&q)[Fmt<FMT>::kQuantBytes / 4], float &dw) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    constexpr int kQW = kQB / 4;
    if constexpr (LAYOUT == kLayoutGguf) {
        // rows are 16-byte multiples, so the block's parity decides its alignment
        load_block_aligned_smem<kQW>(stage, i * nb * kBB + b * kBB, q, dw);
    } else {
        const uint32_t src = stage + static_cast<uint32_t>((i * nb + b) * kQB);
#pragma unroll
        for (int k = 0; k < kQB / 16; ++k) {
            const uint4 t = lds128(src + 16 * k);
            q[4 * k] = t.x;
            q[4 * k + 1] = t.y;
            q[4 * k + 2] = t.z;
            q[4 * k + 3] = t.w;
        }
        const uint32_t h = lds16(stage + static_cast<uint32_t>(tile_rows * nb * kQB + (i * nb + b) * 2));
        dw = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
    }
}

constexpr int kBatchRows = 2;  // rows per row group per iteration

// Reduce-scatter of N values (N = 2, 4, 8, 16 or 32) over the 32 lanes of a warp:
// halving exchanges (lanes with the bit set keep the upper half), then xor sums
// over the remaining lanes. Lane l ends with the warp-wide sum of value
// l >> (5 - log2 N). The association order is fixed, so results are reproducible.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(const float (&v)[N], int lane) {
    static_assert(N == 2 || N == 4 || N == 8 || N == 16 || N == 32, "a power of two <= 32");
    float cur[N];
#pragma unroll
    for (int k = 0; k < N; ++k) cur[k] = v[k];
#pragma unroll
    for (int width = N, bit = 16; width > 1; width >>= 1, bit >>= 1) {
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int k = 0; k < width / 2; ++k) {
            const float send = upper ? cur[k] : cur[width / 2 + k];
            const float keep = upper ? cur[width / 2 + k] : cur[k];
            cur[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = cur[0];
#pragma unroll
    for (int o = 16 / N; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

template <int N> struct Log2;
template <> struct Log2<2> { static constexpr int v = 1; };
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };
template <> struct Log2<32> { static constexpr int v = 5; };

template <int FMT, int LAYOUT, int G, int BPT, int VB, int STAGES>
__global__ void __launch_bounds__(kTmaThreads, (VB >= 8 && FMT == kFmtQ4) ? 2 : 3) dmmv_batch_kernel(const DmmvArgs a) {
    using XV = BVec<FMT>;
    constexpr int kQW = Fmt<FMT>::kQuantBytes / 4;
    constexpr int kGroups = kConsumerThreads / G;          // row groups
    constexpr int kWarpsPerGroup = G >= 32 ? G / 32 : 1;
    constexpr int kLanesPerRow = G >= 32 ? 32 : G;
    constexpr int kN = kBatchRows * VB;                    // partial sums per thread per iteration
    static_assert(G >= 32, "row groups of whole warps");
    static_assert(kN == 2 || kN == 4 || kN == 8 || kN == 16, "2 to 16 partial sums");
    (void)kLanesPerRow;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint8_t *stage0 = smem + kBarrierBytes;
    // per-tile partial sums [pass][iteration][group][warp in group][kN]
    float *red = reinterpret_cast<float *>(stage0 + static_cast<size_t>(STAGES) * a.stage_bytes);

    const int tid = threadIdx.x;
    const int64_t rows = a.rows;
    const int64_t r0 = rows * blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (blockIdx.x + 1) / gridDim.x;
    const int nb = a.nb;
    const int batch = a.batch;

    pdl_launch_dependents();
    if (r1 <= r0) return;
    const uint8_t *w = a.w;
    const int T = a.tile_rows;
    const int ntiles = static_cast<int>((r1 - r0 + T - 1) / T);

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerThreads / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        if (tid != kConsumerThreads) return;
        const uint64_t wpol = l2_evict_first_policy();
        const int npre = ntiles < STAGES ? ntiles : STAGES;
        for (int t = 0; t < npre; ++t) issue_tile<FMT, LAYOUT>(a, w, r0, r1, t, t, stage0, full, wpol);
        int issued = npre;
        bool ok = true;
        for (int t = npre; t < ntiles; ++t) {
            const int s = t % STAGES;
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((t / STAGES) - 1) & 1u)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            issue_tile<FMT, LAYOUT>(a, w, r0, r1, t, s, stage0, full, wpol);
            issued = t + 1;
        }
        if (!ok) atomicOr(a.fault, 1u);
        for (int s = 0; s < STAGES; ++s) {
            const int t_last = (issued - 1 - s) >= 0 ? ((issued - 1 - s) / STAGES) * STAGES + s : -1;
            if (t_last >= 0) (void)mbar_wait(&full[s], static_cast<uint32_t>(t_last / STAGES) & 1u);
        }
        return;
    }

    const int lane = tid & 31;
    const int grp = tid / G;                 // row group
    const int tg = tid % G;                  // thread in the row group
    const int wig = (tid % G) >> 5;          // warp in the row group
    // Block ownership: the first half of the group's threads take the even blocks,
    // the second half the odd ones, so a warp sees one parity (no divergence) and
    // its lanes read rows at a 17-word (Q8_0) / 9-word (Q4_0) stride (no bank
    // conflicts); thread tg owns blocks own_block(tg) + j*G.
    auto own_block = [&](int j) { return 2 * (tg % (G / 2)) + tg / (G / 2) + j * G; };
    pdl_wait();  // activations and outputs may belong to the preceding kernel
    const int npass = (batch + VB - 1) / VB;
    constexpr int kRowsPerIter = kGroups * kBatchRows;
    const int iters = (T + kRowsPerIter - 1) / kRowsPerIter;  // iterations per full tile and pass
    // this pass's vectors, for the blocks this thread owns (kept for the whole
    // launch when one pass covers the batch, reloaded per tile and pass otherwise)
    XV xv[BPT][VB];
    auto load_pass = [&](int pass) {
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            const int b = own_block(j);
#pragma unroll
            for (int v = 0; v < VB; ++v) {
                const int vec = pass * VB + v;
                if (vec < batch) {
                    // straight from global memory (the activation is small and L2-resident)
                    uint32_t xw[8];
                    float dx;
                    load_block_aligned<8>(a.xq, (static_cast<int64_t>(vec) * nb + b) * 34, xw, dx);
                    xv[j][v].set(xw, dx);
                } else {
                    xv[j][v].clear();
                }
            }
        }
    };
    if (npass == 1) load_pass(0);

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
        const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * a.stage_bytes);
        const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
        const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
        for (int pass = 0; pass < npass; ++pass) {
            if (npass > 1) load_pass(pass);
            for (int it = 0; it * kRowsPerIter < nr; ++it) {
                const int base = it * kRowsPerIter;
                float acc[kN];
#pragma unroll
                for (int k = 0; k < kN; ++k) acc[k] = 0.0f;
#pragma unroll
                for (int r = 0; r < kBatchRows; ++r) {
                    const int i = base + r * kGroups + grp;
                    if (i < nr) {
#pragma unroll
                        for (int j = 0; j < BPT; ++j) {
                            const int b = own_block(j);
                            uint32_t wq[kQW];
                            float dw;
                            load_wblock<FMT, LAYOUT>(st, i, b, nb, T, wq, dw);
                            if constexpr (FMT == kFmtQ8) {
#pragma unroll
                                for (int v = 0; v < VB; ++v) {
                                    // vectors past the batch hold zero codes and are never stored
                                    const int sb = xv[j][v].dot(wq);
                                    acc[r * VB + v] = __fmaf_rn(static_cast<float>(sb),
                                                                __fmul_rn(dw, xv[j][v].dx), acc[r * VB + v]);
                                }
                            } else {
                                uint32_t lo[4], hi[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    lo[k] = wq[k] & kLoNib;
                                    hi[k] = wq[k] & kHiNib;
                                }
#pragma unroll
                                for (int v = 0; v < VB; ++v) {
                                    const int sb = xv[j][v].dot(lo, hi);
                                    acc[r * VB + v] = __fmaf_rn(static_cast<float>(sb),
                                                                __fmul_rn(dw, xv[j][v].dx), acc[r * VB + v]);
                                }
                            }
                        }
                    }
                }
                // lane l holds the warp's sum of value (l >> kShift)
                const float part = warp_reduce_scatter<kN>(acc, lane);
                constexpr int kShift = 5 - Log2<kN>::v;
                if ((lane & ((1 << kShift) - 1)) == 0)
                    red[(((pass * iters + it) * kGroups + grp) * kWarpsPerGroup + wig) * kN + (lane >> kShift)] = part;
            }
        }
        // the tile's weights are no longer needed: release the stage first
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        consumer_barrier();
        // combine the warps of each row group, in a fixed order, and store
        const int nout = nr * batch;
        for (int o = tid; o < nout; o += kConsumerThreads) {
            const int vec = o / nr;
            const int i = o - vec * nr;
            const int pass = vec / VB;
            const int v = vec - pass * VB;
            const int it = i / kRowsPerIter;
            const int rem = i - it * kRowsPerIter;
            const int r = rem / kGroups;
            const int g = rem - r * kGroups;
            const float *src = red + (((pass * iters + it) * kGroups + g) * kWarpsPerGroup) * kN + r * VB + v;
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < kWarpsPerGroup; ++q) sum += src[q * kN];
            a.y[static_cast<int64_t>(vec) * a.y_stride + tr0 + i] = sum;
        }
        consumer_barrier();
    }
}

template <int FMT, int LAYOUT, int G, int BPT, int VB, int STAGES>
struct BatchInst {
    static constexpr auto kKernel = &dmmv_batch_kernel<FMT, LAYOUT, G, BPT, VB, STAGES>;
    static int ctas_per_sm(int smem) {
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kKernel, kTmaThreads, static_cast<size_t>(smem)) !=
            cudaSuccess)
            return 1;
        return occ > 0 ? occ : 1;
    }
    static cudaError_t launch(const DmmvArgs &a, int smem, int ctas, cudaStream_t st, bool pdl) {
        static std::atomic<bool> done[64];  // smem limit raised, per device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64 && !done[dev].load(std::memory_order_acquire)) {
            e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kKernel), dev);
            if (e != cudaSuccess) return e;
            done[dev].store(true, std::memory_order_release);
        }
        // never more CTAs than fit in one wave (cached per device and size)
        static std::atomic<uint64_t> occ_cache[64];
        int per_sm = 1;
        const uint64_t c = (dev >= 0 && dev < 64) ? occ_cache[dev].load(std::memory_order_relaxed) : 0;
        if (c != 0 && static_cast<int>(c >> 32) == smem) {
            per_sm = static_cast<int>(c & 0xffffffffu);
        } else {
            per_sm = ctas_per_sm(smem);
            if (dev >= 0 && dev < 64)
                occ_cache[dev].store((static_cast<uint64_t>(smem) << 32) | static_cast<uint32_t>(per_sm),
                                     std::memory_order_relaxed);
        }
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (ctas > sms * per_sm) ctas = sms * per_sm;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
        cfg.blockDim = dim3(kTmaThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kKernel, a);
    }
};

// Variants: (G, BPT, VB) for the widths in use; STAGES 2..4.
template <int FMT, int LAYOUT>
cudaError_t launch_batch_fmt_layout(const DmmvArgs &a, int g, int bpt, int vb, int stages, int smem, int ctas,
                                    cudaStream_t st, bool pdl) {
#define ZDMMV_BVAR(G_, BPT_, VB_, ST_)                                                   \
    if (g == G_ && bpt == BPT_ && vb == VB_ && stages == ST_)                             \
        return BatchInst<FMT, LAYOUT, G_, BPT_, VB_, ST_>::launch(a, smem, ctas, st, pdl);
#define ZDMMV_BVAR_ST(G_, BPT_, VB_) ZDMMV_BVAR(G_, BPT_, VB_, 2) ZDMMV_BVAR(G_, BPT_, VB_, 3) ZDMMV_BVAR(G_, BPT_, VB_, 4)
    ZDMMV_BVAR_ST(128, 1, 2)
    ZDMMV_BVAR_ST(128, 1, 4)
    ZDMMV_BVAR_ST(128, 1, 8)
    ZDMMV_BVAR_ST(128, 2, 2)
    ZDMMV_BVAR_ST(64, 1, 2)
    ZDMMV_BVAR_ST(64, 1, 4)
    ZDMMV_BVAR_ST(64, 1, 8)
    ZDMMV_BVAR_ST(32, 1, 2)
    ZDMMV_BVAR_ST(32, 1, 4)
    ZDMMV_BVAR_ST(32, 1, 8)
    ZDMMV_BVAR_ST(32, 2, 2)
    ZDMMV_BVAR_ST(32, 3, 1)
    ZDMMV_BVAR_ST(32, 4, 1)
#undef ZDMMV_BVAR_ST
#undef ZDMMV_BVAR
    return cudaErrorInvalidConfiguration;
}

template <int FMT>
cudaError_t launch_batch_fmt(const DmmvArgs &a, int layout, int g, int bpt, int vb, int stages, int smem, int ctas,
                             cudaStream_t st, bool pdl) {
    if (layout == kLayoutGguf)
        return launch_batch_fmt_layout<FMT, kLayoutGguf>(a, g, bpt, vb, stages, smem, ctas, st, pdl);
    return launch_batch_fmt_layout<FMT, kLayoutRepacked>(a, g, bpt, vb, stages, smem, ctas, st, pdl);
}

}  // namespace zdmmv
