// zdmmv_mma.cuh -- batched decode DMMV (2..8 activation vectors) on the integer
// tensor cores, GGUF layout, for sm_103a.
//
// With B vectors the DMMV is a thin contraction, rows x B x cols. The dp4a
// kernels spend 8 dp4a per (row, block, vector) on the half-rate integer pipe,
// so at B = 8 they fall behind HBM. Here one mma.sync.m16n8k32.s8.s8.s32 takes a
// block of 16 rows against the same block of all 8 vectors: it is the pages'
// block dot product (the int8x4 dot of "Bringing ZINC to NVIDIA: a CUDA backend",
// int32 accumulation) for 16 x 8 (row, vector) pairs at once, exact by
// construction, and the per-block scales are applied afterwards in fp32 as
// everywhere else (acc = fma(float(s), d_w*d_x, acc)). Q4_0: the nibbles are
// unpacked to bytes 0..15 and the accumulator starts at -8 * sum_i x_i (the -8
// offset of the habr ZINC article, "Что такое DMMV"), so D = sum_i (q_i - 8) x_i.
// The blocks of a row are split over the warps, so the order of the block sums
// differs from the dp4a kernels: results agree with them within the fp32
// tolerance, not bit for bit.
//
// A producer warp streams the weights into a ring of shared-memory stages,
// prefetched before the dependency wait: one 2D tensor copy per stage (16 rows by
// a chunk of blocks, 8-byte elements) whose box is 4 mod 8 words wide, so the 8
// rows of a fragment load fall in 8 distinct bank quads. (Sixteen row-by-row bulk
// copies per stage were measured first: about 50 ns of copy-engine time each kept
// HBM below half its rate.)
//
// Lane (g, t) of a warp (g = lane / 4, t = lane % 4) holds k-slots 4t..4t+3 and
// 16+4t..16+4t+3 of both MMA operands, so the byte -> k-slot assignment is free as
// long as the activation fragment uses the same one. A GGUF block pair (68 or 36
// bytes) is 4-byte aligned; in it the odd block's codes are aligned words and the
// even block's codes start 2 bytes in. Lane t takes aligned words only: for the
// even block the last lane of a quad combines the two stray halves (the first
// two codes, in the word holding the scale, and the last two) with one byte
// permute. The weight words are the A fragments as loaded (Q8_0) or after one
// nibble mask (Q4_0); the activation fragments (the same words of each vector's
// blocks, 256 bytes per block) and a per-block table {accumulator start, d_x} are
// built once per CTA in shared memory from the staged Q8_0 activation.
#pragma once

#include <cuda.h>

#include "zdmmv.h"
#include "zdmmv_mma.h"
#include "zdmmv_tma.cuh"

namespace zdmmv {

constexpr int kMmaRows = 16;        // rows per slab (the MMA's M)
constexpr int kMmaFragBytes = 256;  // per block: 32 lanes x 2 activation words
constexpr int kMmaTableBytes = 64;  // per block: 8 vectors x {accumulator start, d_x}

// 2D tiled tensor copy global -> this CTA's shared memory (box of the map at
// element coordinates x, y; out-of-range elements are zero-filled and counted),
// completing on bar. x * 8 bytes is a multiple of 16; dst is 128-byte aligned.
__device__ __forceinline__ void tensor_copy_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint2 mma_lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// D = A(16x32, s8, row) * B(32x8, s8, col) + C (s32)
__device__ __forceinline__ void mma_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const int (&c)[4]) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(c[0]), "r"(c[1]), "r"(c[2]),
          "r"(c[3]));
}

// Byte permute that finishes lane t's second word of an even block: identity,
// except on the last lane of a quad, which keeps bytes 0, 1 of its word (the
// block's last two codes) and takes bytes 2, 3 of the pair's first word (the
// block's first two codes).
__device__ __forceinline__ uint32_t mma_even_sel(int t) { return t == 3 ? 0x7610u : 0x3210u; }

// One row's weight words of a block pair, for lane t, and both blocks' scales.
// Q8_0: words (k-slots 4t.., 16+4t..) of the even block (ea, eb) and the odd
// block (oa, ob). Q4_0: one word of quant bytes per block (ea, oa); its low
// nibbles fill k-slots 4t.., its high nibbles k-slots 16+4t...
template <int FMT> struct MmaRowPair;

template <> struct MmaRowPair<kFmtQ8> {
    static constexpr int kPairBytes = 68;
    uint32_t ea, eb, oa, ob;
    float d0, d1;
    __device__ __forceinline__ void load(uint32_t row, int t, uint32_t sel) {
        const uint32_t e0 = lds32(row);       // d0 | codes 0, 1
        const uint32_t e8 = lds32(row + 32);  // codes 30, 31 | d1
        ea = lds32(row + 4 + 4 * t);
        eb = __byte_perm(lds32(row + 20 + 4 * t), e0, sel);
        oa = lds32(row + 36 + 4 * t);
        ob = lds32(row + 52 + 4 * t);
        d0 = half_lo(e0);
        d1 = half_hi(e8);
    }
    // A fragments of the even / odd block from rows g and g + 8
    __device__ __forceinline__ static void even(const MmaRowPair &g, const MmaRowPair &h, uint32_t (&a)[4]) {
        a[0] = g.ea;
        a[1] = h.ea;
        a[2] = g.eb;
        a[3] = h.eb;
    }
    __device__ __forceinline__ static void odd(const MmaRowPair &g, const MmaRowPair &h, uint32_t (&a)[4]) {
        a[0] = g.oa;
        a[1] = h.oa;
        a[2] = g.ob;
        a[3] = h.ob;
    }
};

template <> struct MmaRowPair<kFmtQ4> {
    static constexpr int kPairBytes = 36;
    uint32_t ea, oa;
    float d0, d1;
    __device__ __forceinline__ void load(uint32_t row, int t, uint32_t sel) {
        const uint32_t e0 = lds32(row);       // d0 | quant bytes 0, 1
        const uint32_t e4 = lds32(row + 16);  // quant bytes 14, 15 | d1
        ea = __byte_perm(lds32(row + 4 + 4 * t), e0, sel);
        oa = lds32(row + 20 + 4 * t);
        d0 = half_lo(e0);
        d1 = half_hi(e4);
    }
    __device__ __forceinline__ static void frags(uint32_t wg, uint32_t wh, uint32_t (&a)[4]) {
        a[0] = wg & kLoNib;
        a[1] = wh & kLoNib;
        a[2] = (wg >> 4) & kLoNib;
        a[3] = (wh >> 4) & kLoNib;
    }
    __device__ __forceinline__ static void even(const MmaRowPair &g, const MmaRowPair &h, uint32_t (&a)[4]) {
        frags(g.ea, h.ea, a);
    }
    __device__ __forceinline__ static void odd(const MmaRowPair &g, const MmaRowPair &h, uint32_t (&a)[4]) {
        frags(g.oa, h.oa, a);
    }
};

// Activation fragment of block b for lane (g, t) (vector g; zero for g >= batch)
// and, through the quad, the table entry {accumulator start, d_x} of (b, g). The
// lane loads the activation words at the offsets its weight words have
// (activation and weight rows both start 16-byte aligned, so the block
// parities agree). xs: the staged activation, [batch][nb] Q8_0 blocks.
template <int FMT>
__device__ __forceinline__ void mma_build_block(const uint8_t *xs, int nb, int batch, int b, int lane,
                                                uint32_t frag, uint32_t table) {
    const int g = lane >> 2;
    const int t = lane & 3;
    const bool odd = (b & 1) != 0;
    uint32_t r0 = 0u, r1 = 0u;  // codes facing k-slots 4t.. and 16+4t..
    float dx = 0.0f;
    if (g < batch) {
        const uint32_t sel = mma_even_sel(t);
        if constexpr (FMT == kFmtQ8) {
            // the words of the weight pair's loads, taken from the activation pair
            const uint32_t pb = smem_addr(xs) + static_cast<uint32_t>((g * nb + (b & ~1)) * 34);
            if (!odd) {
                const uint32_t e0 = lds32(pb);
                r0 = lds32(pb + 4 + 4 * t);
                r1 = __byte_perm(lds32(pb + 20 + 4 * t), e0, sel);
                dx = half_lo(e0);
            } else {
                r0 = lds32(pb + 36 + 4 * t);
                r1 = lds32(pb + 52 + 4 * t);
                dx = half_hi(lds32(pb + 32));
            }
        } else {
            // Q4_0 quant byte j of lane t faces activation codes j and j + 16
            const uint32_t xb = smem_addr(xs) + static_cast<uint32_t>((g * nb + b) * 34);
            if (!odd) {
                r0 = __byte_perm(lds32(xb + 4 + 4 * t), lds32(xb), sel);
                r1 = __byte_perm(lds32(xb + 20 + 4 * t), lds32(xb + 16), sel);
                dx = half_lo(lds32(xb));
            } else {
                r0 = lds32(xb + 2 + 4 * t);
                r1 = lds32(xb + 18 + 4 * t);
                dx = half_hi(lds32(xb - 2));
            }
        }
    }
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(frag + static_cast<uint32_t>(lane * 8)), "r"(r0), "r"(r1)
                 : "memory");
    // Q4_0: the accumulator starts at -8 times the block's code sum (quad sum)
    int sx = FMT == kFmtQ4 ? dp4a_ss(r0, kOnes, dp4a_ss(r1, kOnes, 0)) : 0;
    if constexpr (FMT == kFmtQ4) {
        sx += __shfl_xor_sync(0xffffffffu, sx, 1);
        sx += __shfl_xor_sync(0xffffffffu, sx, 2);
    }
    if (t == 0) {
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(table + static_cast<uint32_t>(g * 8)),
                     "r"(static_cast<uint32_t>(-8 * sx)), "r"(__float_as_uint(dx))
                     : "memory");
    }
}

template <int NW>
__device__ __forceinline__ void mma_consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// One block's MMA and fp32 update. f: the activation words, tab: {c[2t], dx[2t],
// c[2t+1], dx[2t+1]} (c: accumulator start), dg, dh: the block's scales of rows
// g and g + 8.
__device__ __forceinline__ void mma_block(const uint32_t (&a)[4], const uint2 &f, const uint4 &tab, float dg,
                                          float dh, float (&acc)[4]) {
    const int c[4] = {static_cast<int>(tab.x), static_cast<int>(tab.z), static_cast<int>(tab.x),
                      static_cast<int>(tab.z)};
    int d[4];
    mma_16832(d, a, f.x, f.y, c);
    const float dx0 = __uint_as_float(tab.y);
    const float dx1 = __uint_as_float(tab.w);
    acc[0] = __fmaf_rn(__int2float_rn(d[0]), __fmul_rn(dg, dx0), acc[0]);
    acc[1] = __fmaf_rn(__int2float_rn(d[1]), __fmul_rn(dg, dx1), acc[1]);
    acc[2] = __fmaf_rn(__int2float_rn(d[2]), __fmul_rn(dh, dx0), acc[2]);
    acc[3] = __fmaf_rn(__int2float_rn(d[3]), __fmul_rn(dh, dx1), acc[3]);
}

// NW consumer warps + 1 producer warp; one CTA per SM (shared memory).
// CTA c takes slabs c, c + gridDim.x, ...; each slab (16 rows) streams in
// a.nchunks stages of a.cb blocks per row. wmap: the weight rows as a 2D tensor
// of 8-byte elements, box {a.pitch / 8, 16}.
template <int FMT, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32, 1) dmmv_mma_kernel(const MmaArgs a,
                                                                    const __grid_constant__ CUtensorMap wmap) {
    using RP = MmaRowPair<FMT>;
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kConsumers = NW * 32;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xbar = empty + STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kBarrierBytes - 8);
    uint8_t *xs = smem + kBarrierBytes;  // staged activation, later the partial sums
    uint8_t *frag = xs + a.x_region;
    uint8_t *table = frag + static_cast<size_t>(a.nb) * kMmaFragBytes;
    uint8_t *stage0 = table + static_cast<size_t>(a.nb) * kMmaTableBytes;
    const int stage_bytes = kMmaRows * a.pitch;

    const int tid = threadIdx.x;
    const int64_t nslabs = (a.rows + kMmaRows - 1) / kMmaRows;
    const int my_slabs = blockIdx.x < nslabs
                             ? static_cast<int>((nslabs - 1 - blockIdx.x) / gridDim.x + 1)
                             : 0;
    const int items = my_slabs * a.nchunks;

    pdl_launch_dependents();
    if (items == 0) return;
    // tensor copies land on 128-byte boundaries (the host plan keeps every stage
    // offset a multiple of 128; this guards the base)
    if ((smem_addr(stage0) & 127u) != 0u) {
        if (tid == 0) atomicOr(a.fault, ZDMMV_FAULT_SMEM_ALIGN);
        return;
    }

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumers) {
        // ------------------------------------------------------- producer
        if (tid != kConsumers) return;
        const uint64_t wpol = l2_evict_first_policy();
        auto issue = [&](int it) {
            const int s = it % STAGES;
            const int64_t slab = blockIdx.x + static_cast<int64_t>(it / a.nchunks) * gridDim.x;
            const int k = it % a.nchunks;
            // the whole box counts, rows and columns past the matrix included (zero-filled)
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
            tensor_copy_2d(stage0 + static_cast<size_t>(s) * stage_bytes, &wmap, k * a.cb * kBB / 8,
                           static_cast<int>(slab * kMmaRows), &full[s], wpol);
        };
        const int npre = items < STAGES ? items : STAGES;
        for (int it = 0; it < npre; ++it) issue(it);
        int issued = npre;
        pdl_wait();  // the activations may be written by the preceding kernel
        {
            const uint32_t xbytes = static_cast<uint32_t>(a.batch) * static_cast<uint32_t>(a.nb) * 34u;
            mbar_arrive_expect_tx(xbar, xbytes);
            bulk_copy_g2s(xs, a.xq, xbytes, xbar, l2_evict_last_policy());
        }
        bool ok = true;
        for (int it = npre; it < items; ++it) {
            const int s = it % STAGES;
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((it / STAGES) - 1) & 1u)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            issue(it);
            issued = it + 1;
        }
        if (!ok) atomicOr(a.fault, 1u);
        // no copy may still be in flight when the CTA exits
        for (int s = 0; s < STAGES; ++s) {
            const int t_last = (issued - 1 - s) >= 0 ? ((issued - 1 - s) / STAGES) * STAGES + s : -1;
            if (t_last >= 0) (void)mbar_wait(&full[s], static_cast<uint32_t>(t_last / STAGES) & 1u);
        }
        (void)mbar_wait(xbar, 0);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint32_t sel = mma_even_sel(t);
    pdl_wait();  // outputs may still be read by the preceding kernel
    // A timed-out wait marks the CTA aborted: the warps skip all further waits and
    // work but keep meeting at the consumer barrier, so no warp is left waiting.
    bool ok = __all_sync(0xffffffffu, mbar_wait(xbar, 0));
    if (!ok) {
        if (lane == 0) atomicOr(a.fault, 1u);
        *abort_flag = 1;
    } else {
        for (int b = warp; b < a.nb; b += NW)
            mma_build_block<FMT>(xs, a.nb, a.batch, b,  lane,
                                 smem_addr(frag) + static_cast<uint32_t>(b * kMmaFragBytes),
                                 smem_addr(table) + static_cast<uint32_t>(b * kMmaTableBytes));
    }
    mma_consumer_barrier<NW>();  // fragments and table complete; xs is free from here on

    const uint32_t frag_a = smem_addr(frag) + static_cast<uint32_t>(lane * 8);
    const uint32_t table_a = smem_addr(table) + static_cast<uint32_t>(t * 16);
    const uint32_t red_a = smem_addr(xs);
    int it = 0;
    for (int si = 0; si < my_slabs; ++si) {
        const int64_t r0 = (blockIdx.x + static_cast<int64_t>(si) * gridDim.x) * kMmaRows;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int k = 0; k < a.nchunks; ++k, ++it) {
            const int s = it % STAGES;
            if (ok && __any_sync(0xffffffffu, *abort_flag != 0)) ok = false;
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(it / STAGES) & 1u));
                if (!ok) {
                    if (lane == 0) atomicOr(a.fault, 1u);
                    *abort_flag = 1;
                }
            }
            if (!ok) continue;
            const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * stage_bytes);
            const uint32_t rowg = st + static_cast<uint32_t>(g * a.pitch);
            const uint32_t rowh = rowg + static_cast<uint32_t>(8 * a.pitch);
            const int cbk = min(a.cb, a.nb - k * a.cb);
            const int np = cbk >> 1;
            const int b00 = k * a.cb;  // first block of the chunk
#pragma unroll 4
            for (int p = warp; p < np; p += NW) {
                const uint32_t off = static_cast<uint32_t>(p * RP::kPairBytes);
                RP wg, wh;
                wg.load(rowg + off, t, sel);
                wh.load(rowh + off, t, sel);
                const int b0 = b00 + 2 * p;
                const uint2 f0 = mma_lds64(frag_a + static_cast<uint32_t>(b0 * kMmaFragBytes));
                const uint2 f1 = mma_lds64(frag_a + static_cast<uint32_t>((b0 + 1) * kMmaFragBytes));
                const uint4 t0 = lds128(table_a + static_cast<uint32_t>(b0 * kMmaTableBytes));
                const uint4 t1 = lds128(table_a + static_cast<uint32_t>((b0 + 1) * kMmaTableBytes));
                uint32_t a[4];
                RP::even(wg, wh, a);
                mma_block(a, f0, t0, wg.d0, wh.d0, acc);
                RP::odd(wg, wh, a);
                mma_block(a, f1, t1, wg.d1, wh.d1, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // combine the warps' partial sums (double-buffered: one barrier per slab)
        const uint32_t red = red_a + static_cast<uint32_t>((si & 1) * NW * 512);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(red + static_cast<uint32_t>(warp * 512 + lane * 16)),
                     "f"(acc[0]), "f"(acc[1]), "f"(acc[2]), "f"(acc[3])
                     : "memory");
        mma_consumer_barrier<NW>();
        if (tid < kMmaRows * 8 && !*abort_flag) {
            const int v = tid >> 4;
            const int r = tid & 15;
            const uint32_t e = static_cast<uint32_t>((((r & 7) * 4 + (v >> 1)) * 4 + (r >> 3) * 2 + (v & 1)) * 4);
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < NW; ++w) sum += __uint_as_float(lds32(red + static_cast<uint32_t>(w * 512) + e));
            if (v < a.batch && r0 + r < a.rows) a.y[static_cast<int64_t>(v) * a.y_stride + r0 + r] = sum;
        }
    }
}

template <int FMT, int NW, int STAGES>
struct MmaInst {
    static constexpr auto kKernel = &dmmv_mma_kernel<FMT, NW, STAGES>;
    static cudaError_t launch(const MmaArgs &a, const CUtensorMap &wmap, int smem_bytes, cudaStream_t st, bool pdl) {
        static std::atomic<bool> done[64];  // smem limit raised, per device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!done[dev].load(std::memory_order_acquire)) {
            e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kKernel), dev);
            if (e != cudaSuccess) return e;
            done[dev].store(true, std::memory_order_release);
        }
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t nslabs = (a.rows + kMmaRows - 1) / kMmaRows;
        const int64_t ctas = nslabs < sms ? nslabs : sms;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
        cfg.blockDim = dim3((NW + 1) * 32, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kKernel, a, wmap);
    }
};

template <int FMT>
cudaError_t launch_mma_fmt(const MmaArgs &a, const CUtensorMap &wmap, const MmaPlan &p, cudaStream_t st,
                           bool pdl) {
#define ZDMMV_MMA(NW_, S_) \
    if (p.warps == NW_ && p.stages == S_) return MmaInst<FMT, NW_, S_>::launch(a, wmap, p.smem_bytes, st, pdl);
    ZDMMV_MMA(8, 2)
    ZDMMV_MMA(8, 3)
    ZDMMV_MMA(8, 4)
    ZDMMV_MMA(8, 5)
    ZDMMV_MMA(8, 6)
    ZDMMV_MMA(16, 2)
    ZDMMV_MMA(16, 3)
    ZDMMV_MMA(16, 4)
    ZDMMV_MMA(16, 5)
    ZDMMV_MMA(16, 6)
#undef ZDMMV_MMA
    return cudaErrorInvalidConfiguration;
}

}  // namespace zdmmv
