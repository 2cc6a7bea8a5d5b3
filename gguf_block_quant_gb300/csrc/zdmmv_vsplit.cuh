// zdmmv_vsplit.cuh -- batched decode DMMV (2..8 activation vectors, one weight
// stream) with the vectors split over the consumer warps, for sm_103a.
//
// The weight tiles stream through the TMA ring exactly as in the single-vector
// kernel (producer warp, full/empty mbarriers, tiles prefetched before the
// dependency wait), so HBM sees the weights once per call. The 4 consumer warps
// form NVG vector groups; each warp holds V activation vectors in registers
// (the single-vector kernel's block-pair registers, V times) and the warps of a
// vector group split the tile's rows. Every warp of the CTA reads the same
// shared-memory tile (NVG reads per tile), loads each weight pair once for its V
// vectors, and reduces each (row, vector) with the single-vector kernel's
// xor-shuffle tree; no cross-warp combine, no barrier inside the tile loop.
//
// Per lane and vector the arithmetic is the single-vector kernel's, in the same
// order (its pairs, then the same reduction tree), so each vector's
// result is bitwise the one zdmmv_q{8,4}_0 returns for it.
#pragma once

#include "zdmmv_tma.cuh"

namespace zdmmv {

// The weight words of one block pair of one staged row, held in registers.
template <int FMT, int LAYOUT> struct PairW;

template <int FMT> struct PairW<FMT, kLayoutGguf> {
    static constexpr int kW = Pair<FMT, kLayoutGguf>::kWords;
    uint32_t r[kW];
    // row: shared-memory address of the staged row; p: pair index
    __device__ __forceinline__ void load(uint32_t row, uint32_t /*scales*/, int p) {
        const uint32_t a = row + static_cast<uint32_t>(p * RowGeom<FMT, kLayoutGguf>::kPairBytes);
#pragma unroll
        for (int k = 0; k < kW; ++k) r[k] = lds32(a + 4 * k);
    }
    __device__ __forceinline__ float dwa() const { return half_lo(r[0]); }
    __device__ __forceinline__ float dwb() const { return FMT == kFmtQ8 ? half_hi(r[8]) : half_hi(r[4]); }
};

template <int FMT> struct PairW<FMT, kLayoutRepacked> {
    using P = Pair<FMT, kLayoutRepacked>;
    static constexpr int kW = P::kWords;
    uint32_t r[kW];
    uint32_t ws;
    // row: address of the row's quant words; scales: address of its scale array.
    // The chunks are loaded in the pair's rotated order (Pair::rotation), the
    // order the lane's activation words are held in.
    __device__ __forceinline__ void load(uint32_t row, uint32_t scales, int p) {
        const uint32_t a = row + static_cast<uint32_t>(p * RowGeom<FMT, kLayoutRepacked>::kPairQuantBytes);
        const int rot = P::rotation(p);
#pragma unroll
        for (int k = 0; k < P::kChunks; ++k) {
            const uint4 t = lds128(a + 16u * static_cast<uint32_t>(k ^ rot));
            r[4 * k] = t.x;
            r[4 * k + 1] = t.y;
            r[4 * k + 2] = t.z;
            r[4 * k + 3] = t.w;
        }
        ws = lds32(scales + 4 * p);
    }
    __device__ __forceinline__ float dwa() const { return half_lo(ws); }
    __device__ __forceinline__ float dwb() const { return half_hi(ws); }
};

// acc = fma(sA, dwA*dxA, acc); acc = fma(sB, dwB*dxB, acc): Pair::fma_pair's
// update with the weights already in registers.
template <int FMT, int LAYOUT>
__device__ __forceinline__ float pair_update(const Pair<FMT, LAYOUT> &x, const PairW<FMT, LAYOUT> &w, float acc) {
    int sa, sb;
    x.sums(w.r, sa, sb);
    acc = __fmaf_rn(static_cast<float>(sa), __fmul_rn(w.dwa(), x.dxa), acc);
    acc = __fmaf_rn(static_cast<float>(sb), __fmul_rn(w.dwb(), x.dxb), acc);
    return acc;
}

// a.batch vectors of Q8_0 blocks, contiguous at a.xq (staged in shared memory by
// one bulk copy); outputs at a.y + v * a.y_stride. FX = true: the consumers
// quantize the fp32 activations a.xf ([batch][cols], contiguous) into the same
// shared-memory blocks themselves (the stand-alone quantizer's bytes), so the
// results are those of the quantizer followed by the batched call.
template <int FMT, int LAYOUT, int LPR, int PPL, int V, int NVG, int STAGES, bool FX = false>
__global__ void __launch_bounds__(kTmaThreads, 3) dmmv_vsplit_kernel(const DmmvArgs a) {
    using P = Pair<FMT, LAYOUT>;
    using W = PairW<FMT, LAYOUT>;
    constexpr int kWarps = kConsumerThreads / 32;
    static_assert(kWarps % NVG == 0, "vector groups split the consumer warps evenly");
    constexpr int kRowWarps = kWarps / NVG;                // warps sharing one vector group
    constexpr int kGroupsPerWarp = 32 / LPR;               // row groups per warp
    constexpr int kRowGroups = kRowWarps * kGroupsPerWarp; // row groups per vector group
    constexpr int kRowsIlp = 2;                            // rows in flight per row group
    constexpr int kN = kRowsIlp * V;                       // sums per lane per iteration

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xbar = empty + STAGES;
    uint8_t *xs = smem + kBarrierBytes;  // the batch's Q8_0 activation blocks, one bulk copy
    uint8_t *stage0 = xs + a.x_bytes_padded;

    const int tid = threadIdx.x;
    const int64_t rows = a.rows;
    const int64_t r0 = rows * blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (blockIdx.x + 1) / gridDim.x;
    const int nb = a.nb;

    pdl_launch_dependents();
    if (r1 <= r0) return;
    const int T = a.tile_rows;
    const int ntiles = static_cast<int>((r1 - r0 + T - 1) / T);

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        // ------------------------------------------------------- producer
        if (tid != kConsumerThreads) return;
        const uint64_t wpol = l2_evict_first_policy();
        // one tile before the dependency wait, then the activation copy, then the
        // rest of the ring (this CTA's copies are served in issue order)
        const int nring = ntiles < STAGES ? ntiles : STAGES;
        issue_tile<FMT, LAYOUT>(a, a.w, r0, r1, 0, 0, stage0, full, wpol);
        int issued = 1;
        pdl_wait();  // the activations may be written by the preceding kernel
        if constexpr (!FX) {
            const uint32_t xbytes = static_cast<uint32_t>(a.batch) * static_cast<uint32_t>(nb) * 34u;
            mbar_arrive_expect_tx(xbar, xbytes);
            bulk_copy_g2s(xs, a.xq, xbytes, xbar, l2_evict_last_policy());
        }
        for (; issued < nring; ++issued) issue_tile<FMT, LAYOUT>(a, a.w, r0, r1, issued, issued, stage0, full, wpol);
        bool ok = true;
        for (int t = issued; t < ntiles; ++t) {
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
        if constexpr (!FX) (void)mbar_wait(xbar, 0);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int vg = warp % NVG;                                   // vector group
    const int rg = (warp / NVG) * kGroupsPerWarp + lane / LPR;   // row group within it
    const int l = lane % LPR;
    const int npairs = nb >> 1;
    const bool full_pairs = npairs == LPR * PPL;  // every lane owns PPL pairs of every row
    pdl_wait();  // outputs may still be read, and the activations written, by the preceding kernel
    if constexpr (FX) {
        // nb is a multiple of 8 on this path: whole quads of blocks per vector
        quantize_quads_to_smem<kWarps, 8, true>(a.xf, a.batch * (nb >> 2), xs, warp, lane);
        consumer_barrier();
    } else {
        // waits are warp-uniform so a timeout can never split a warp before its shuffles
        if (!__all_sync(0xffffffffu, mbar_wait(xbar, 0))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
    }
    // this warp's vectors, from the staged activation blocks
    P xr[V][PPL];
    bool live[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int vec = vg * V + v;
        live[v] = vec < a.batch;
        const uint32_t xv = smem_addr(xs) + static_cast<uint32_t>((live[v] ? vec : 0) * nb * 34);
#pragma unroll
        for (int j = 0; j < PPL; ++j) {
            const int p = owned_pair<LPR>(l, j);
            uint32_t w17[17];
            if (p < npairs) {
                load_x_pair_words_smem(xv, p, w17);
            } else {
#pragma unroll
                for (int k = 0; k < 17; ++k) w17[k] = 0;
            }
            xr[v][j].set(w17, p);
        }
    }

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
        const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * a.stage_bytes);
        const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
        const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
        for (int base = 0; base < nr; base += kRowGroups * kRowsIlp) {
            float acc[kRowsIlp][V];
#pragma unroll
            for (int r = 0; r < kRowsIlp; ++r) {
#pragma unroll
                for (int v = 0; v < V; ++v) acc[r][v] = 0.0f;
            }
            // the shared-memory addresses of row r of this chunk (quants; scales in the repacked layout)
            const auto row_addr = [&](int i, uint32_t &row, uint32_t &scales) {
                if constexpr (LAYOUT == kLayoutGguf) {
                    row = st + static_cast<uint32_t>(i * nb * Fmt<FMT>::kBlockBytes);
                    scales = 0;
                } else {
                    row = st + static_cast<uint32_t>(i * nb * Fmt<FMT>::kQuantBytes);
                    scales = st + static_cast<uint32_t>(T * nb * Fmt<FMT>::kQuantBytes + i * nb * 2);
                }
            };
            if (LAYOUT == kLayoutGguf && full_pairs && base + kRowGroups * kRowsIlp <= nr) {
                // every row of the chunk and every pair of the lane exists: no predicates, so
                // the rows' loads can be issued together (the same updates in the same order;
                // measured: Q8_0 14336 x 4096, B = 2 / 4 / 8, 11.2 / 12.1 / 15.9 -> 10.9 / 11.8 /
                // 15.3 us; the repacked layout's two-row weight registers spill, so it keeps the
                // predicated loop)
#pragma unroll
                for (int j = 0; j < PPL; ++j) {
                    const int p = owned_pair<LPR>(l, j);
                    W w[kRowsIlp];
#pragma unroll
                    for (int r = 0; r < kRowsIlp; ++r) {
                        uint32_t row, scales;
                        row_addr(base + r * kRowGroups + rg, row, scales);
                        w[r].load(row, scales, p);
                    }
#pragma unroll
                    for (int r = 0; r < kRowsIlp; ++r) {
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[r][v] = pair_update(xr[v][j], w[r], acc[r][v]);
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < kRowsIlp; ++r) {
                    const int i = base + r * kRowGroups + rg;
                    if (i < nr) {
                        uint32_t row, scales;
                        row_addr(i, row, scales);
#pragma unroll
                        for (int j = 0; j < PPL; ++j) {
                            const int p = owned_pair<LPR>(l, j);
                            if (p < npairs) {
                                W w;
                                w.load(row, scales, p);
#pragma unroll
                                for (int v = 0; v < V; ++v) acc[r][v] = pair_update(xr[v][j], w, acc[r][v]);
                            }
                        }
                    }
                }
            }
            // the kN sums land on lanes 0, LPR/kN, ... of the group (value index r*V + v)
            float flat[kN];
#pragma unroll
            for (int r = 0; r < kRowsIlp; ++r) {
#pragma unroll
                for (int v = 0; v < V; ++v) flat[r * V + v] = acc[r][v];
            }
            const float part = group_reduce_scatter<LPR, kN>(flat, l);
            constexpr int kSpan = LPR / kN;
            if (l % kSpan == 0) {
                const int idx = l / kSpan;
                const int r = idx / V;
                const int v = idx % V;
                const int i = base + r * kRowGroups + rg;
                const int vec = vg * V + v;
                if (i < nr && vec < a.batch) a.y[static_cast<int64_t>(vec) * a.y_stride + tr0 + i] = part;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

template <int FMT, int LAYOUT, int LPR, int PPL, int V, int NVG, int STAGES, bool FX>
struct VsplitInst {
    static constexpr auto kKernel = &dmmv_vsplit_kernel<FMT, LAYOUT, LPR, PPL, V, NVG, STAGES, FX>;
    // one wave of the CTAs that fit (occupancy cached per device and size)
    static cudaError_t launch(const DmmvArgs &a, const TmaPlan &p, int max_per_sm, cudaStream_t st, bool pdl) {
        static std::atomic<bool> done[64];  // smem limit raised, per device
        static std::atomic<uint64_t> occ_cache[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!done[dev].load(std::memory_order_acquire)) {
            e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kKernel), dev);
            if (e != cudaSuccess) return e;
            done[dev].store(true, std::memory_order_release);
        }
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
        if (max_per_sm > 0 && per_sm > max_per_sm) per_sm = max_per_sm;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        int64_t ctas = static_cast<int64_t>(sms) * per_sm;
        if (ctas > a.rows) ctas = a.rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
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

// p.lpr / p.ppl as in the single-vector plan; v vectors per warp, nvg groups; p.stages 2 or 3.
template <int FMT, int LAYOUT, bool FX>
cudaError_t launch_vsplit_layout(const DmmvArgs &a, const TmaPlan &p, int v, int nvg, int max_per_sm,
                                 cudaStream_t st, bool pdl) {
#define ZDMMV_VS(LPR_, PPL_, V_, NVG_)                                                                        \
    if (p.lpr == LPR_ && p.ppl == PPL_ && v == V_ && nvg == NVG_)                                             \
        return p.stages == 3 ? VsplitInst<FMT, LAYOUT, LPR_, PPL_, V_, NVG_, 3, FX>::launch(a, p, max_per_sm, st, pdl) \
                             : VsplitInst<FMT, LAYOUT, LPR_, PPL_, V_, NVG_, 2, FX>::launch(a, p, max_per_sm, st, pdl);
#define ZDMMV_VS_ALL(LPR_, PPL_) \
    ZDMMV_VS(LPR_, PPL_, 1, 2) ZDMMV_VS(LPR_, PPL_, 1, 4) ZDMMV_VS(LPR_, PPL_, 2, 1) ZDMMV_VS(LPR_, PPL_, 2, 2) \
    ZDMMV_VS(LPR_, PPL_, 2, 4)
    ZDMMV_VS_ALL(8, 1)
    ZDMMV_VS_ALL(16, 1)
    ZDMMV_VS_ALL(32, 1)
    ZDMMV_VS_ALL(32, 2)
    ZDMMV_VS(32, 4, 1, 2)
    ZDMMV_VS(32, 4, 1, 4)
#undef ZDMMV_VS_ALL
#undef ZDMMV_VS
    return cudaErrorInvalidConfiguration;
}

template <int FMT, bool FX>
cudaError_t launch_vsplit_fmt(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                              cudaStream_t st, bool pdl) {
    if (layout == kLayoutGguf) return launch_vsplit_layout<FMT, kLayoutGguf, FX>(a, p, v, nvg, max_per_sm, st, pdl);
    return launch_vsplit_layout<FMT, kLayoutRepacked, FX>(a, p, v, nvg, max_per_sm, st, pdl);
}

}  // namespace zdmmv
