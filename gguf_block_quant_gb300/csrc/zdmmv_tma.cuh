// zdmmv_tma.cuh -- the TMA-pipelined decode DMMV kernel for sm_103a.
//
// Design (one CTA = 4 consumer warps + 1 producer warp, several CTAs per SM):
//  * Each CTA owns a contiguous range of rows. In GGUF layout consecutive rows
//    are consecutive bytes, so a tile of T rows is ONE contiguous chunk and is
//    fetched with a single bulk TMA copy (cp.async.bulk) into a shared-memory
//    stage; the repacked layout takes one copy for the quants and one for the
//    scales. The weight stream is read from HBM exactly once, with an
//    evict-first L2 policy (it is never re-read).
//  * The producer lane keeps STAGES tiles in flight (full/empty mbarrier pairs);
//    the 4 consumer warps never wait on global memory, only on a stage.
//  * The Q8_0 activation (at most a few KB) is staged once per CTA by one more
//    bulk copy and then held in REGISTERS: lane l of a row group owns PPL block
//    pairs (owned_pair) for every row, so the inner loop reads only weights
//    from shared memory (the pages stage the input vector in LDS so that the
//    weights own the cache: habr ZINC article, "Трюк с shared memory"; here the
//    activation goes one level further, into registers).
//  * LPR lanes share a row; their partial sums meet in an xor-shuffle tree
//    (subgroupAdd -> __shfl reductions: "CUDA backend for ZINC", "4. Kernel port
//    strategy"). The reduction order depends only on the row's contents, never
//    on its position, so results are bitwise invariant under row permutation
//    and identical for the same row in any call.
//  * Every mbarrier wait is bounded (1 s); on a timeout the kernel sets the
//    device fault word, drains its own copies (bounded) and returns.
#pragma once

#include <atomic>

#include "zdmmv_device.cuh"
#include "zdmmv_internal.h"

namespace zdmmv {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int FMT, int LAYOUT> struct RowGeom;
template <int FMT> struct RowGeom<FMT, kLayoutGguf> {
    static constexpr int kPairBytes = 2 * Fmt<FMT>::kBlockBytes;
};
template <int FMT> struct RowGeom<FMT, kLayoutRepacked> {
    static constexpr int kPairQuantBytes = 2 * Fmt<FMT>::kQuantBytes;
};

// One lane's contribution to one row: its pairs (owned_pair) in order j = 0..PPL-1.
// stage: shared-memory address of the tile.
template <int FMT, int LAYOUT, int LPR, int PPL>
__device__ __forceinline__ float row_partial(const Pair<FMT, LAYOUT> (&xr)[PPL], uint32_t stage, int i,
                                             int tile_rows, int nb, int l) {
    const int npairs = nb >> 1;
    float acc = 0.0f;
    if constexpr (LAYOUT == kLayoutGguf) {
        constexpr int kW = Pair<FMT, LAYOUT>::kWords;
        const uint32_t row = stage + static_cast<uint32_t>(i * nb * Fmt<FMT>::kBlockBytes);
#pragma unroll
        for (int j = 0; j < PPL; ++j) {
            const int p = owned_pair<LPR>(l, j);
            if (p < npairs) {
                const uint32_t w = row + static_cast<uint32_t>(p * RowGeom<FMT, LAYOUT>::kPairBytes);
                uint32_t r[kW];
#pragma unroll
                for (int k = 0; k < kW; ++k) r[k] = lds32(w + 4 * k);
                acc = xr[j].fma_w(r, acc);
            }
        }
    } else {
        const uint32_t rq = stage + static_cast<uint32_t>(i * nb * Fmt<FMT>::kQuantBytes);
        const uint32_t rs = stage + static_cast<uint32_t>(tile_rows * nb * Fmt<FMT>::kQuantBytes + i * nb * 2);
#pragma unroll
        for (int j = 0; j < PPL; ++j) {
            const int p = owned_pair<LPR>(l, j);
            if (p < npairs) {
                const uint32_t ws = lds32(rs + 4 * p);
                acc = xr[j].fma_pair(rq + p * RowGeom<FMT, LAYOUT>::kPairQuantBytes, ws, acc);
            }
        }
    }
    return acc;
}

// The contributions of one lane to N rows i0, i0 + step, ... of a GGUF tile whose
// rows and this lane's pairs all exist: every row's weight words of pair j are
// loaded before any of them is used, then each row takes row_partial's updates in
// row_partial's order (so the sums are the same bits).
template <int FMT, int LPR, int PPL, int N>
__device__ __forceinline__ void rows_partial_full(const Pair<FMT, kLayoutGguf> (&xr)[PPL], uint32_t stage, int i0,
                                                  int step, int nb, int l, float (&acc)[N]) {
    constexpr int kW = Pair<FMT, kLayoutGguf>::kWords;
    const uint32_t row_bytes = static_cast<uint32_t>(nb * Fmt<FMT>::kBlockBytes);
#pragma unroll
    for (int r = 0; r < N; ++r) acc[r] = 0.0f;
#pragma unroll
    for (int j = 0; j < PPL; ++j) {
        const uint32_t pofs = static_cast<uint32_t>(owned_pair<LPR>(l, j) * RowGeom<FMT, kLayoutGguf>::kPairBytes);
        uint32_t w[N][kW];
#pragma unroll
        for (int r = 0; r < N; ++r) {
            const uint32_t a = stage + static_cast<uint32_t>(i0 + r * step) * row_bytes + pofs;
#pragma unroll
            for (int k = 0; k < kW; ++k) w[r][k] = lds32(a + 4 * k);
        }
#pragma unroll
        for (int r = 0; r < N; ++r) acc[r] = xr[j].fma_w(w[r], acc[r]);
    }
}

// Bytes of tile t of a CTA's row range [r0, r1).
template <int FMT>
__device__ __forceinline__ uint32_t tile_bytes(const DmmvArgs &a, int64_t r0, int64_t r1, int t) {
    const int64_t tr0 = r0 + static_cast<int64_t>(t) * a.tile_rows;
    const int nr = static_cast<int>(min(static_cast<int64_t>(a.tile_rows), r1 - tr0));
    return static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.nb) * Fmt<FMT>::kBlockBytes;
}

// Bulk copy (or copies, repacked layout) of tile t of matrix w into dst,
// completing on bar; the caller has already announced the bytes.
template <int FMT, int LAYOUT>
__device__ __forceinline__ void copy_tile(const DmmvArgs &a, const uint8_t *w, int64_t r0, int64_t r1, int t,
                                          uint8_t *dst, uint64_t *bar, uint64_t pol) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kQB = Fmt<FMT>::kQuantBytes;
    const int T = a.tile_rows;
    const int nb = a.nb;
    const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
    const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
    if constexpr (LAYOUT == kLayoutGguf) {
        bulk_copy_g2s(dst, w + tr0 * nb * kBB, static_cast<uint32_t>(nr) * static_cast<uint32_t>(nb) * kBB, bar, pol);
    } else {
        const uint32_t qbytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(nb) * kQB;
        const uint32_t sbytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(nb) * 2u;
        bulk_copy_g2s(dst, w + tr0 * nb * kQB, qbytes, bar, pol);
        bulk_copy_g2s(dst + static_cast<size_t>(T) * nb * kQB, w + a.rows * nb * kQB + tr0 * nb * 2, sbytes, bar,
                      pol);
    }
}

// Issue tile t into stage s (and, with a second matrix w2, the same rows of w2
// into the stage's second half).
template <int FMT, int LAYOUT>
__device__ __forceinline__ void issue_tile(const DmmvArgs &a, const uint8_t *w, int64_t r0, int64_t r1, int t, int s,
                                           uint8_t *stage0, uint64_t *full, uint64_t pol,
                                           const uint8_t *w2 = nullptr) {
    uint8_t *dst = stage0 + static_cast<size_t>(s) * a.stage_bytes;
    const uint32_t bytes = tile_bytes<FMT>(a, r0, r1, t);
    mbar_arrive_expect_tx(&full[s], w2 ? 2 * bytes : bytes);
    copy_tile<FMT, LAYOUT>(a, w, r0, r1, t, dst, &full[s], pol);
    if (w2) copy_tile<FMT, LAYOUT>(a, w2, r0, r1, t, dst + a.stage_bytes / 2, &full[s], pol);
}

__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// FX = true: the kernel reads the fp32 activation (a.xf) and quantizes it to
// Q8_0 blocks in shared memory itself (same device function as the stand-alone
// quantizer, hence identical bytes), instead of staging a.xq.
// Argmax epilogue ordering: a larger value wins, equal values keep the smaller row.
__device__ __forceinline__ bool argmax_better(float v, int row, float bv, int brow) {
    return row >= 0 && (brow < 0 || v > bv || (v == bv && row < brow));
}

// EPI = 0: store y. EPI = 1 (argmax epilogue): keep each row group's running
// (max, first row) in registers, reduce over the CTA and store one 8-byte partial
// per CTA in a.argmax_parts; no y is written. EPI = 2 (accumulate epilogue):
// y = fma(s, W.x, y) with s = sigmoid(*a.gate), or s = 1 without a gate.
// EPI = 3 (SwiGLU pair): a.w is the gate matrix (stack) and a.w_b the up matrix
// (stack) of the same shape; each stage holds the tile's gate rows then the same
// rows of up, the row group computes a gate row and its up row as its two rows
// in flight, and y = silu(gate . x) * (up . x) is stored.
template <int FMT, int LAYOUT, int LPR, int PPL, int STAGES, int MINB, bool FX, int EPI = 0>
__global__ void __launch_bounds__(kTmaThreads, MINB) dmmv_tma_kernel(const DmmvArgs a) {
    using P = Pair<FMT, LAYOUT>;
    constexpr int kRowsPar = kConsumerThreads / LPR;
    constexpr int kRowsIlp = kTmaRowsIlp;
    static_assert(kConsumerThreads % LPR == 0 && LPR <= 32, "row groups must live inside a warp");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xbar = empty + STAGES;
    uint8_t *xs = smem + kBarrierBytes;
    uint8_t *stage0 = xs + a.x_bytes_padded;

    const int tid = threadIdx.x;
    const int slot = blockIdx.y;
    const int64_t rows = a.rows;
    const int64_t r0 = rows * blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (blockIdx.x + 1) / gridDim.x;
    const int nb = a.nb;

    // Dependent launches may start as soon as every CTA of this grid is resident;
    // what they do before their own dependency wait is stream weights only. A
    // gather that waits for its index list lets them start only after that wait:
    // then the list is complete whenever a later launch starts, and a later
    // gather of the same selection may read it at once (a.idx_ready).
    const bool early_idx = a.idx != nullptr && a.idx_ready != 0;
    if (a.idx == nullptr || early_idx) pdl_launch_dependents();

    // a second stack (e.g. the up projections next to the gates) takes the slots
    // from slots_a on, with the same selected experts and activations
    const bool second = EPI != 3 && a.w_b != nullptr && slot >= a.slots_a;
    const int sel = second ? slot - a.slots_a : slot;
    float *y = (second ? a.y_b : a.y) + sel * a.y_stride;
    const uint8_t *w = second ? a.w_b : a.w;
    const uint8_t *w_up = EPI == 3 ? a.w_b : nullptr;  // SwiGLU pair: the up matrix
    if (a.idx != nullptr) {
        int e;
        if (early_idx) {
            e = __ldcg(a.idx + sel);  // complete since an earlier gather's wait; L2, not a stale L1 line
        } else {
            pdl_wait();  // the index list may be written by the preceding kernel
            e = a.idx[sel];
            pdl_launch_dependents();
        }
        if (e < 0 || e >= a.n_experts) {
            if (early_idx) pdl_wait();  // y may still be read by the preceding kernel
            for (int64_t r = r0 + tid; r < r1; r += blockDim.x) y[r] = __int_as_float(0x7fc00000);
            if (tid == 0 && a.status != nullptr) atomicExch(a.status, 1);
            return;
        }
        w += static_cast<int64_t>(e) * a.expert_stride;
        if (EPI == 3) w_up += static_cast<int64_t>(e) * a.expert_stride;
    }
    if (r1 <= r0) {
        if constexpr (EPI == 1) {
            if (tid == 0) a.argmax_parts[blockIdx.x] = make_uint2(0u, 0xffffffffu);  // no candidate
        }
        return;
    }
    const int T = a.tile_rows;
    const int ntiles = static_cast<int>((r1 - r0 + T - 1) / T);

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerThreads / 32);
        }
        mbar_init(xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        // ------------------------------------------------------- producer
        if (tid != kConsumerThreads) return;
        const uint64_t wpol = l2_evict_first_policy();
        // Weights are read-only parameters: the first tile streams before waiting
        // for the preceding kernel, overlapping its tail. The activation copy goes
        // next and the rest of the ring after it: this CTA's copies are served in
        // issue order, and no tile can be used before the activation (the whole
        // ring ahead of it: dense Q4_0 4096^2 chain 3.16 us, LM head 43.8 us, Q8_0
        // 14336 x 4096 10.0 us; one tile: 3.01, 43.4, 9.75 us).
        const int nring = ntiles < STAGES ? ntiles : STAGES;
        issue_tile<FMT, LAYOUT>(a, w, r0, r1, 0, 0, stage0, full, wpol, w_up);
        int issued = 1;
        pdl_wait();
        if constexpr (!FX) {
            const uint32_t xbytes = static_cast<uint32_t>(nb) * 34u;
            mbar_arrive_expect_tx(xbar, xbytes);
            bulk_copy_g2s(xs, a.xq + sel * a.xq_stride, xbytes, xbar, l2_evict_last_policy());
        }
        for (; issued < nring; ++issued)
            issue_tile<FMT, LAYOUT>(a, w, r0, r1, issued, issued, stage0, full, wpol, w_up);
        bool ok = true;
        for (int t = issued; t < ntiles; ++t) {
            const int s = t % STAGES;
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((t / STAGES) - 1) & 1u)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            issue_tile<FMT, LAYOUT>(a, w, r0, r1, t, s, stage0, full, wpol, w_up);
            issued = t + 1;
        }
        if (!ok) atomicOr(a.fault, 1u);
        // Never leave while a copy into this CTA's shared memory is in flight:
        // wait (bounded) for the last copy issued into every stage.
        for (int s = 0; s < STAGES; ++s) {
            const int t_last = (issued - 1 - s) >= 0 ? ((issued - 1 - s) / STAGES) * STAGES + s : -1;
            if (t_last >= 0) (void)mbar_wait(&full[s], static_cast<uint32_t>(t_last / STAGES) & 1u);
        }
        if constexpr (!FX) (void)mbar_wait(xbar, 0);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int g = tid / LPR;  // row group
    const int l = tid % LPR;  // lane inside the row group
    pdl_wait();               // outputs may still be read, and the activation written, by the preceding kernel
    const bool full_pairs = (nb >> 1) == LPR * PPL;  // every lane owns PPL pairs of every row
    if constexpr (FX) {
        // quantize the fp32 activation into Q8_0 blocks in shared memory (nb is a
        // multiple of 8 on this path)
        quantize_quads_to_smem<kConsumerThreads / 32>(a.xf + sel * a.xf_stride, nb >> 2, xs, tid >> 5, lane);
        consumer_barrier();
    } else {
        // waits are made warp-uniform so a timeout can never split a warp before its shuffles
        if (!__all_sync(0xffffffffu, mbar_wait(xbar, 0))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
    }
    P xr[PPL];
#pragma unroll
    for (int j = 0; j < PPL; ++j) {
        const int p = owned_pair<LPR>(l, j);
        if (p < (nb >> 1)) {
            uint32_t v[17];
            load_x_pair_words_smem(smem_addr(xs), p, v);
            xr[j].set(v, p);
        }
    }

    float scale = 1.0f;  // accumulate epilogue: the gate's sigmoid
    if constexpr (EPI == 2) {
        if (a.gate != nullptr) scale = 1.0f / (1.0f + expf(-*a.gate));
    }
    float best = 0.0f;  // argmax epilogue: this row group's running maximum and its row
    int best_row = -1;
    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
            if (lane == 0) atomicOr(a.fault, 1u);
            return;
        }
        const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * a.stage_bytes);
        const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
        const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
        if constexpr (EPI == 3) {
            // a gate row and the same up row in flight; then silu(gate) * up
            const uint32_t st_up = st + static_cast<uint32_t>(a.stage_bytes / 2);
            for (int base = 0; base < nr; base += kRowsPar) {
                const int i = base + g;
                float gv = 0.0f, uv = 0.0f;
                if (i < nr) {
                    gv = row_partial<FMT, LAYOUT, LPR, PPL>(xr, st, i, T, nb, l);
                    uv = row_partial<FMT, LAYOUT, LPR, PPL>(xr, st_up, i, T, nb, l);
                }
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) {
                    gv += __shfl_xor_sync(0xffffffffu, gv, o);
                    uv += __shfl_xor_sync(0xffffffffu, uv, o);
                }
                if (l == 0 && i < nr) y[tr0 + i] = __fmul_rn(__fdiv_rn(gv, 1.0f + expf(-gv)), uv);
            }
        } else {
            // kRowsIlp rows per row group at a time: independent loads, dot chains and
            // shuffle trees interleave; every row still gets the same reduction tree
            for (int base = 0; base < nr; base += kRowsPar * kRowsIlp) {
                float acc[kRowsIlp];
                if constexpr (LAYOUT == kLayoutGguf) {
                    if (full_pairs && base + kRowsPar * kRowsIlp <= nr) {
                        rows_partial_full<FMT, LPR, PPL, kRowsIlp>(xr, st, base + g, kRowsPar, nb, l, acc);
                    } else {
#pragma unroll
                        for (int r = 0; r < kRowsIlp; ++r) {
                            const int i = base + r * kRowsPar + g;
                            acc[r] = i < nr ? row_partial<FMT, LAYOUT, LPR, PPL>(xr, st, i, T, nb, l) : 0.0f;
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < kRowsIlp; ++r) {
                        const int i = base + r * kRowsPar + g;
                        acc[r] = i < nr ? row_partial<FMT, LAYOUT, LPR, PPL>(xr, st, i, T, nb, l) : 0.0f;
                    }
                }
                if constexpr (EPI == 0) {
                    // the rows' sums land on lanes 0, LPR/kRowsIlp, ... of the group
                    const float part = group_reduce_scatter<LPR, kRowsIlp>(acc, l);
                    constexpr int kSpan = LPR / kRowsIlp;
                    const int i = base + (l / kSpan) * kRowsPar + g;
                    if (l % kSpan == 0 && i < nr) y[tr0 + i] = part;
                } else {
#pragma unroll
                    for (int o = LPR / 2; o > 0; o >>= 1) {
#pragma unroll
                        for (int r = 0; r < kRowsIlp; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
                    }
#pragma unroll
                    for (int r = 0; r < kRowsIlp; ++r) {
                        const int i = base + r * kRowsPar + g;
                        if constexpr (EPI == 2) {
                            if (l == 0 && i < nr) y[tr0 + i] = __fmaf_rn(scale, acc[r], y[tr0 + i]);
                        } else {
                            // rows reach a row group in increasing order: a strictly larger value replaces
                            if (i < nr && (best_row < 0 || acc[r] > best)) {
                                best = acc[r];
                                best_row = static_cast<int>(tr0 + i);
                            }
                        }
                    }
                }
            }
        }  // EPI != 3
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if constexpr (EPI == 1) {
        // reduce the row groups' candidates (kept on every lane of a group) in group order
        __shared__ float cand_v[kRowsPar];
        __shared__ int cand_r[kRowsPar];
        if (l == 0) {
            cand_v[g] = best;
            cand_r[g] = best_row;
        }
        consumer_barrier();
        if (tid == 0) {
            float bv = 0.0f;
            int br = -1;
            for (int q = 0; q < kRowsPar; ++q)
                if (argmax_better(cand_v[q], cand_r[q], bv, br)) {
                    bv = cand_v[q];
                    br = cand_r[q];
                }
            a.argmax_parts[blockIdx.x] = make_uint2(__float_as_uint(bv), static_cast<uint32_t>(br));
        }
    }
}

// ------------------------------------------------------------------ host side
template <int FMT, int LAYOUT, int LPR, int PPL, int STAGES, bool FX, int EPI = 0>
struct TmaInst {
    static constexpr int kMinBlocks = PPL >= 4 ? 2 : 4;
    static constexpr auto kKernel = &dmmv_tma_kernel<FMT, LAYOUT, LPR, PPL, STAGES, kMinBlocks, FX, EPI>;
    static void *fn() { return reinterpret_cast<void *>(kKernel); }

    static cudaError_t prepare() {
        // raise the dynamic shared-memory limit once per device
        static std::atomic<bool> done[64];  // smem limit raised, per device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
        e = raise_dynamic_smem_limit(fn(), dev);
        if (e != cudaSuccess) return e;
        if (dev < 64) done[dev].store(true, std::memory_order_release);
        return cudaSuccess;
    }

    static cudaError_t launch(const DmmvArgs &a, const TmaPlan &p, int ctas_per_slot, int slots, cudaStream_t st,
                              bool pdl) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
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

    // CTAs per SM for this shared-memory size; the occupancy query is cached per
    // device (one entry: a decode stream calls the same shapes over and over)
    static int ctas_per_sm(int smem_bytes) {
        static std::atomic<uint64_t> cache[64];  // (smem_bytes << 32) | occupancy, per device
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return 1;
        const bool cacheable = dev >= 0 && dev < 64;
        if (cacheable) {
            const uint64_t c = cache[dev].load(std::memory_order_relaxed);
            if (c != 0 && static_cast<int>(c >> 32) == smem_bytes) return static_cast<int>(c & 0xffffffffu);
        }
        if (prepare() != cudaSuccess) return 1;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kKernel, kTmaThreads,
                                                          static_cast<size_t>(smem_bytes)) != cudaSuccess)
            return 1;
        occ = occ > 0 ? occ : 1;
        if (cacheable)
            cache[dev].store((static_cast<uint64_t>(smem_bytes) << 32) | static_cast<uint32_t>(occ),
                             std::memory_order_relaxed);
        return occ;
    }
};

// Dispatch over the (lpr, ppl, stages) variants instantiated for one format.
template <int FMT, int LAYOUT, bool FX, int EPI = 0, typename F>
cudaError_t with_variant(const TmaPlan &p, F &&f) {
#define ZDMMV_VARIANT(LPR_, PPL_, ST_)                                        \
    if (p.lpr == LPR_ && p.ppl == PPL_ && p.stages == ST_)                    \
        return f(TmaInst<FMT, LAYOUT, LPR_, PPL_, ST_, FX, EPI>{});
    ZDMMV_VARIANT(8, 1, 4)
    ZDMMV_VARIANT(16, 1, 4)
    ZDMMV_VARIANT(32, 1, 4)
    ZDMMV_VARIANT(32, 2, 4)
    ZDMMV_VARIANT(32, 4, 4)
    ZDMMV_VARIANT(8, 1, 3)
    ZDMMV_VARIANT(16, 1, 3)
    ZDMMV_VARIANT(32, 1, 3)
    ZDMMV_VARIANT(32, 2, 3)
    ZDMMV_VARIANT(32, 4, 3)
    ZDMMV_VARIANT(8, 1, 2)
    ZDMMV_VARIANT(16, 1, 2)
    ZDMMV_VARIANT(32, 1, 2)
    ZDMMV_VARIANT(32, 2, 2)
    ZDMMV_VARIANT(32, 4, 2)
#undef ZDMMV_VARIANT
    return cudaErrorInvalidConfiguration;
}

template <int FMT>
cudaError_t launch_tma_fmt(const DmmvArgs &a, const TmaPlan &p, int layout, bool fused_x, int ctas_per_slot,
                           int slots, cudaStream_t st, bool pdl) {
    auto go = [&](auto inst) { return decltype(inst)::launch(a, p, ctas_per_slot, slots, st, pdl); };
    if (fused_x) {
        if (layout == kLayoutGguf) return with_variant<FMT, kLayoutGguf, true>(p, go);
        return with_variant<FMT, kLayoutRepacked, true>(p, go);
    }
    if (layout == kLayoutGguf) return with_variant<FMT, kLayoutGguf, false>(p, go);
    return with_variant<FMT, kLayoutRepacked, false>(p, go);
}

template <int FMT, int EPI>
cudaError_t launch_epi_fmt(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl,
                           int slots = 1) {
    auto go = [&](auto inst) { return decltype(inst)::launch(a, p, ctas, slots, st, pdl); };
    if (layout == kLayoutGguf) return with_variant<FMT, kLayoutGguf, false, EPI>(p, go);
    return with_variant<FMT, kLayoutRepacked, false, EPI>(p, go);
}

template <int FMT>
cudaError_t launch_argmax_fmt(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl) {
    return launch_epi_fmt<FMT, 1>(a, p, layout, ctas, st, pdl);
}

template <int FMT, int EPI = 0>
int tma_ctas_per_sm_fmt(int layout, const TmaPlan &p) {
    int occ = 1;
    auto q = [&](auto inst) {
        occ = decltype(inst)::ctas_per_sm(p.smem_bytes);
        return cudaSuccess;
    };
    if (layout == kLayoutGguf)
        (void)with_variant<FMT, kLayoutGguf, false, EPI>(p, q);
    else
        (void)with_variant<FMT, kLayoutRepacked, false, EPI>(p, q);
    return occ;
}

}  // namespace zdmmv
