// zdmmv_bmma.cuh -- batched decode DMMV (up to 8 Q8_0 activation vectors) on the
// fp16 tensor cores, GGUF layout, for sm_103a.
//
// With B vectors the DMMV is a thin contraction, rows x B x cols: the pages' block
// dot product (the int8x4 dot of "Bringing ZINC to NVIDIA: a CUDA backend", int32
// block sums, then the two fp16 scales) for every (row, vector) pair. The dp4a
// kernels spend 8 dp4a per (row, block, vector), so at 8 vectors they are bound by
// instruction issue, not HBM. Here one block of 16 rows meets the same block of
// all 8 vectors in two mma.sync.m16n8k16 (fp16 in, fp32 accumulation):
//  * a weight code becomes an fp16 value with one or two logic operations and no
//    subtraction: Q8_0 code c as 1152 + c (the offset byte c + 128 under the fp16
//    exponent of 1024), a Q4_0 low nibble n as 1024 + n = 1032 + (n - 8), a high
//    nibble as 1024 + 16 n = 1152 + 16 (n - 8) with the activation code it meets
//    divided by 16 (exact in fp16);
//  * the offsets are taken out by the accumulator's start value, per block and
//    vector: -1152 * sum(x) (Q8_0), -(1032 * sum(x_low) + 72 * sum(x_high)) (Q4_0);
//  * every product is an integer (or, for the Q4_0 high nibbles, 16 times an
//    integer divided by 16), and every partial sum is an integer below 2^24 in
//    magnitude (Q8_0: 32 * 1280 * 128 + 1152 * 32 * 128 < 10^7), so the block sum
//    D is exact: the int32 block sum of the pages, as an fp32 value;
//  * y[r, v] += D * (d_w[r] * d_x[v]) in fp32, one fma per (row, vector, block).
// The blocks of a row are split over 8 warps whose partial sums are added in a
// fixed order at the end, so results are reproducible but the order of the fp32
// sums differs from the single-vector kernel: they agree with it within the fp32
// tolerance, not bit for bit.
//
// The weights stream as in the fp32-activation tensor-core kernel: a producer warp
// issues one 2D tensor copy per stage (32 rows = two 16-row slabs, by a chunk of 32
// blocks) into a ring of stages, the first before the dependency wait; the
// staged row pitch is 4 mod 8 words, so the fragment loads of the 8 rows of a lane
// quad hit distinct banks. Warp w takes slab w / 8 of each stage and blocks
// 4 (w % 8) .. 4 (w % 8) + 3 of the chunk; its lane t loads the aligned words of
// each block pair that the other tensor-core kernels load (at immediate offsets).
// The activation fragments (512 bytes per block: lane (g, t) of a consumer warp
// reads the codes of vector g facing its weight slots) and a per-block table {d_x,
// accumulator start} per vector are built once per CTA from the Q8_0 activation,
// which the producer bulk-copies after the dependency wait into the top of the
// fragment region (one request stream per CTA: 4-byte loads from global memory by
// all the consumer warps of every CTA took ~3 us at 8 vectors); the consumers
// load it into registers, meet at a barrier, and write the fragments over it, so
// every stage of the ring streams weights from the start.
#pragma once

#include "zdmmv_xf32_mma.cuh"

namespace zdmmv {

struct BmmaArgs {
    const uint8_t *w;    // GGUF rows
    const uint8_t *xq;   // Q8_0 activation of vector 0; vector v at xq + v * xq_stride
    const float *xf;     // FX: fp32 activations [batch][nb * 32], quantized by the kernel
    float *y;            // output of vector 0; vector v at y + v * y_stride
    uint32_t *fault;     // device fault word
    int64_t rows;
    int64_t xq_stride;   // bytes between vectors' activations
    int64_t y_stride;    // floats between vectors' outputs
    int32_t nb;          // blocks per row
    int32_t batch;       // 1..8
    int32_t nchunks;     // stages per 32-row group (chunks of kBmChunkBlocks blocks)
    int32_t pitch;       // shared-memory bytes per staged row (4 mod 8 words)
    int32_t red_bufs;    // 1 or 2 buffers of warp partial sums
};

constexpr int kBmWarps = 16;                             // consumer warps
constexpr int kBmSlabs = 2;                              // 16-row slabs per stage
constexpr int kBmParts = kBmWarps / kBmSlabs;            // warps sharing a slab (8)
constexpr int kBmWarpBlocks = 4;                         // blocks per warp and stage
constexpr int kBmChunkBlocks = kBmParts * kBmWarpBlocks; // blocks per row and stage (32)
constexpr int kBmGroupRows = kBmSlabs * kMmaRows;        // rows per stage (32)
constexpr int kBmFragBytes = 512;                        // per block: 32 lanes x 8 fp16 codes
constexpr int kBmTableBytes = 64;                        // per block: 8 vectors x {d_x, start}
constexpr int kBmRedBytes = kBmWarps * 512;              // one buffer of warp partial sums
constexpr int kBmMaxBlocks = 128;                        // blocks per row (4096 columns) at most

// fp16 pairs of the int8 codes in bytes (0, 2) and (1, 3) of r, exact.
__device__ __forceinline__ void bm_code_pairs(uint32_t r, uint32_t &p02, uint32_t &p13) {
    constexpr uint32_t k1152 = 0x64806480u;  // fp16 1152 = 1024 + 128
    const uint32_t u = r ^ 0x80808080u;
    p02 = h2_sub(__byte_perm(u, 0x64646464u, 0x4240u), k1152);
    p13 = h2_sub(__byte_perm(u, 0x64646464u, 0x4341u), k1152);
}
// The same pairs divided by 16 (exact: the codes have at most 8 significant bits).
__device__ __forceinline__ void bm_code_pairs16(uint32_t r, uint32_t &p02, uint32_t &p13) {
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16
    constexpr uint32_t kMinus72 = 0xD480D480u;    // fp16 -72 = -1152 / 16
    const uint32_t u = r ^ 0x80808080u;
    p02 = h2_fma(__byte_perm(u, 0x64646464u, 0x4240u), kSixteenth, kMinus72);
    p13 = h2_fma(__byte_perm(u, 0x64646464u, 0x4341u), kSixteenth, kMinus72);
}

// The two activation words of block b of a vector staged at xv (shared memory)
// for lane t, holding the codes that face the lane's weight words (XmRow, in
// zdmmv_xf32_mma.cuh: Q8_0, the words at the offsets of the weight pair's loads;
// Q4_0, the codes that the low nibbles of the lane's quant word meet, then those
// the high nibbles meet), and the block's d_x. xv is 4-byte
// aligned and holds whole blocks; every load stays inside blocks b & ~1 .. b | 1
// of the vector (nb is even). The lanes of a warp may hold blocks of both
// parities: both take the same loads at offsets chosen by parity and the same
// selects, so the warp does not diverge.
template <int FMT>
__device__ __forceinline__ void bm_load_x(uint32_t xv, int b, int t, uint32_t sel, uint32_t &r0, uint32_t &r1,
                                          float &dx) {
    const bool odd = (b & 1) != 0;
    if constexpr (FMT == kFmtQ8) {
        // even block: d | codes 0, 1 at the pair's start, codes 2 + 4t.., 18 + 4t.. (the
        // last lane's second word completed from the first); odd block: codes 4t..,
        // 16 + 4t.. of the second block, its scale in the word at 32
        const uint32_t pb = xv + static_cast<uint32_t>((b & ~1) * 34) + static_cast<uint32_t>(4 * t);
        const uint32_t e = lds32(xv + static_cast<uint32_t>((b & ~1) * 34 + (odd ? 32 : 0)));
        const uint32_t w0 = lds32(pb + (odd ? 36u : 4u));
        const uint32_t w1 = lds32(pb + (odd ? 52u : 20u));
        r0 = w0;
        r1 = odd ? w1 : __byte_perm(w1, e, sel);
        dx = odd ? half_hi(e) : half_lo(e);
    } else {
        // even block (4-byte aligned): d | codes 0, 1, then codes 2 + 4t.. and 18 + 4t..
        // (the last lane completed from the words at 0 and 16); odd block: codes 4t..
        // and 16 + 4t.. are aligned, its scale in the word before it
        const uint32_t xb = xv + static_cast<uint32_t>(b * 34);
        const uint32_t e = lds32(odd ? xb - 2 : xb);
        const uint32_t h = lds32(xb + (odd ? 14u : 16u));  // used by even blocks; 4-byte aligned either way
        const uint32_t w0 = lds32(xb + static_cast<uint32_t>(4 * t) + (odd ? 2u : 4u));
        const uint32_t w1 = lds32(xb + static_cast<uint32_t>(4 * t) + (odd ? 18u : 20u));
        r0 = odd ? w0 : __byte_perm(w0, e, sel);
        r1 = odd ? w1 : __byte_perm(w1, h, sel);
        dx = odd ? half_hi(e) : half_lo(e);
    }
}

// Fragment slot `slot` = 4 v + t (16 bytes at slot * 16) of block b and, through
// the quad of lanes holding its four slots t, the table entry {d_x, accumulator
// start} of vector v (at v * 8), from the lane's activation words; zeros give the
// slots of vectors past the batch and of blocks past the row.
template <int FMT>
__device__ __forceinline__ void bm_store_block(uint32_t r0, uint32_t r1, float dx, int slot, uint32_t frag,
                                               uint32_t table) {
    uint32_t f[4];
    bm_code_pairs(r0, f[0], f[1]);
    if constexpr (FMT == kFmtQ4) {
        bm_code_pairs16(r1, f[2], f[3]);
    } else {
        bm_code_pairs(r1, f[2], f[3]);
    }
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(frag + static_cast<uint32_t>(slot * 16)),
                 "r"(f[0]), "r"(f[1]), "r"(f[2]), "r"(f[3])
                 : "memory");
    // code sums of the quad (the block's 32 codes): r0's codes, r1's codes
    int s0 = dp4a_ss(r0, kOnes, 0);
    int s1 = dp4a_ss(r1, kOnes, 0);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    // the weights' offsets (Q8_0: 1152 on every code; Q4_0: 1032 on the codes facing
    // low nibbles, 72 on those facing high nibbles), exact integers in fp32
    const int start = FMT == kFmtQ8 ? -1152 * (s0 + s1) : -(1032 * s0 + 72 * s1);
    // table entry of the vector pair (2i, 2i + 1): {d_x[2i], d_x[2i+1], start[2i], start[2i+1]}
    if ((slot & 3) == 0) {
        const int v = slot >> 2;
        const uint32_t e = table + static_cast<uint32_t>((v >> 1) * 16 + (v & 1) * 4);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(e), "f"(dx) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(e + 8), "f"(static_cast<float>(start)) : "memory");
    }
}

// A fragments of one block from the lane's weight words, the codes with their
// offsets (no subtraction): rows g and g + 8, register order {row g, row g + 8} x
// {k-pair (2t, 2t+1), k-pair (2t+8, 2t+9)}.
template <int FMT> struct BmFrags;
template <> struct BmFrags<kFmtQ4> {
    __device__ __forceinline__ static void make(uint32_t wg, uint32_t wh, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
        constexpr uint32_t kMagic = 0x64006400u;  // fp16 1024, both halves
        const uint32_t sg = wg >> 8, sh = wh >> 8;
        a0[0] = (wg & 0x000F000Fu) | kMagic;
        a0[1] = (wh & 0x000F000Fu) | kMagic;
        a0[2] = (sg & 0x000F000Fu) | kMagic;
        a0[3] = (sh & 0x000F000Fu) | kMagic;
        a1[0] = (wg & 0x00F000F0u) | kMagic;
        a1[1] = (wh & 0x00F000F0u) | kMagic;
        a1[2] = (sg & 0x00F000F0u) | kMagic;
        a1[3] = (sh & 0x00F000F0u) | kMagic;
    }
};
template <> struct BmFrags<kFmtQ8> {
    __device__ __forceinline__ static void pairs(uint32_t w, uint32_t &p02, uint32_t &p13) {
        const uint32_t u = w ^ 0x80808080u;
        p02 = __byte_perm(u, 0x64646464u, 0x4240u);
        p13 = __byte_perm(u, 0x64646464u, 0x4341u);
    }
    __device__ __forceinline__ static void make(uint32_t ag, uint32_t bg, uint32_t ah, uint32_t bh, uint32_t (&a0)[4],
                                                uint32_t (&a1)[4]) {
        pairs(ag, a0[0], a0[2]);
        pairs(ah, a0[1], a0[3]);
        pairs(bg, a1[0], a1[2]);
        pairs(bh, a1[1], a1[3]);
    }
};

// Packed fp32 pairs (sm_100 family): {a0, a1} = {x0, x1} * {y0, y1} and
// {a0, a1} = fma({x0, x1}, {y0, y1}, {a0, a1}), each lane of the pair the IEEE
// round-to-nearest operation of the scalar instruction.
__device__ __forceinline__ void f2_mul(float &a0, float &a1, float x0, float x1, float y0, float y1) {
    asm("{\n\t.reg .b64 ra, rx, ry;\n\tmov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
        "mul.rn.f32x2 ra, rx, ry;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(a0), "=f"(a1)
        : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
__device__ __forceinline__ void f2_fma(float &a0, float &a1, float x0, float x1, float y0, float y1) {
    asm("{\n\t.reg .b64 ra, rx, ry;\n\tmov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
        "mov.b64 ra, {%0, %1};\n\tfma.rn.f32x2 ra, rx, ry, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// One block: two MMAs from the accumulator start, then the fp32 update of the
// lane's four (row, vector) sums, acc += D * (d_w * d_x) (one rounding for the
// product of the scales, one for the fma). tab = {d_x[2t], d_x[2t+1], start[2t],
// start[2t+1]}; dg, dh: the block's scales of rows g and g + 8.
__device__ __forceinline__ void bm_block(const uint32_t (&a0)[4], const uint32_t (&a1)[4], const uint4 &f,
                                         const uint4 &tab, float dg, float dh, float (&acc)[4]) {
    const float c0 = __uint_as_float(tab.z), c1 = __uint_as_float(tab.w);
    const float c[4] = {c0, c1, c0, c1};
    float d[4];
    mma_16816(d, a0, f.x, f.y, c);
    mma_16816(d, a1, f.z, f.w, d);
    const float dx0 = __uint_as_float(tab.x), dx1 = __uint_as_float(tab.y);
    float pg0, pg1, ph0, ph1;
    f2_mul(pg0, pg1, dg, dg, dx0, dx1);
    f2_mul(ph0, ph1, dh, dh, dx0, dx1);
    f2_fma(acc[0], acc[1], d[0], d[1], pg0, pg1);
    f2_fma(acc[2], acc[3], d[2], d[3], ph0, ph1);
}

// Pair P (blocks 2P, 2P + 1 of the warp's four) for this lane: rows g (rg, rgt)
// and g + 8 (rh, rht), fb / tb: the fragment and table addresses of the warp's
// first block for this lane. A stage loads both pairs' operands first, then
// computes them.
template <int FMT> struct BmPair {
    XmRow<FMT> wg, wh;
    uint4 f0, f1, t0, t1;
};
template <int FMT, int P>
__device__ __forceinline__ void bm_pair_load(BmPair<FMT> &d, uint32_t rg, uint32_t rgt, uint32_t rh, uint32_t rht,
                                             uint32_t fb, uint32_t tb, uint32_t sel) {
    constexpr int kF = 2 * P * kBmFragBytes;
    constexpr int kT = 2 * P * kBmTableBytes;
    d.wg.template load<P>(rg, rgt, sel);
    d.wh.template load<P>(rh, rht, sel);
    d.f0 = ldsi128<kF>(fb);
    d.f1 = ldsi128<kF + kBmFragBytes>(fb);
    d.t0 = ldsi128<kT>(tb);
    d.t1 = ldsi128<kT + kBmTableBytes>(tb);
}
template <int FMT>
__device__ __forceinline__ void bm_pair_compute(const BmPair<FMT> &d, float (&acc)[4]) {
    uint32_t a0[4], a1[4];
    if constexpr (FMT == kFmtQ4) {
        BmFrags<kFmtQ4>::make(d.wg.ea, d.wh.ea, a0, a1);
        bm_block(a0, a1, d.f0, d.t0, d.wg.d0, d.wh.d0, acc);
        BmFrags<kFmtQ4>::make(d.wg.oa, d.wh.oa, a0, a1);
        bm_block(a0, a1, d.f1, d.t1, d.wg.d1, d.wh.d1, acc);
    } else {
        BmFrags<kFmtQ8>::make(d.wg.ea, d.wg.eb, d.wh.ea, d.wh.eb, a0, a1);
        bm_block(a0, a1, d.f0, d.t0, d.wg.d0, d.wh.d0, acc);
        BmFrags<kFmtQ8>::make(d.wg.oa, d.wg.ob, d.wh.oa, d.wh.ob, a0, a1);
        bm_block(a0, a1, d.f1, d.t1, d.wg.d1, d.wh.d1, acc);
    }
}

__device__ __forceinline__ void bm_consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kBmWarps * 32) : "memory");
}

// kBmWarps consumer warps + 1 producer warp, one CTA per SM. CTA c takes the
// 32-row groups c, c + gridDim.x, ..., each in a.nchunks stages of kBmChunkBlocks
// blocks per row. wmap: the weight rows as a 2D tensor of 8-byte elements, box
// {a.pitch / 8, kBmGroupRows}.
// FX = true: the consumers quantize the fp32 activations (a.xf) into the staged
// Q8_0 blocks themselves, with the stand-alone quantizer's arithmetic
// (quantize_quads_to_smem), so the results are the bits of the quantizer followed
// by the FX = false kernel.
template <int FMT, int STAGES, bool FX>
__global__ void __launch_bounds__((kBmWarps + 1) * 32, 1) dmmv_bmma_kernel(const BmmaArgs a,
                                                                          const __grid_constant__ CUtensorMap wmap) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kConsumers = kBmWarps * 32;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xbar = empty + STAGES;  // the staged activation has landed
    uint64_t *xready = xbar + 1;      // FX: the activation is quantized (its loads are done)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kBarrierBytes - 8);
    const int nb_pad = a.nchunks * kBmChunkBlocks;
    uint8_t *frag = smem + kBarrierBytes;
    uint8_t *table = frag + static_cast<size_t>(nb_pad) * kBmFragBytes;
    uint8_t *red = table + static_cast<size_t>(nb_pad) * kBmTableBytes;
    uint8_t *stage0 = red + static_cast<size_t>(a.red_bufs) * kBmRedBytes;
    const int stage_bytes = kBmGroupRows * a.pitch;
    // The activation is staged at the top of the fragment region (which holds 512
    // bytes per block, the staged activation at most 8 x 34 + 16 per block): every
    // consumer loads its share into registers, and after a barrier the fragments
    // overwrite it, so the whole ring is free for weights from the start. Vector v
    // at xs + v * x_pitch: a Q8_0 row plus 16 bytes (4 mod 32 words), so the 8
    // vectors' words of one block fall in distinct banks (FX: the quantizer writes
    // the rows back to back).
    const int x_row = a.nb * 34;
    const int x_pitch = FX ? x_row : x_row + 16;
    uint8_t *xs = frag + (static_cast<size_t>(nb_pad) * kBmFragBytes - static_cast<size_t>(a.batch) * x_pitch);

    const int tid = threadIdx.x;
    const int64_t ngroups = (a.rows + kBmGroupRows - 1) / kBmGroupRows;
    const int my_groups = blockIdx.x < ngroups ? static_cast<int>((ngroups - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    const int items = my_groups * a.nchunks;

    pdl_launch_dependents();
    if (items == 0) return;
    // tensor copies land on 128-byte boundaries (the host plan keeps every offset
    // a multiple of 128; this guards the base)
    if ((smem_addr(stage0) & 127u) != 0u) {
        if (tid == 0) atomicOr(a.fault, ZDMMV_FAULT_SMEM_ALIGN);
        return;
    }

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBmWarps);
        }
        mbar_init(xbar, 1);
        mbar_init(xready, 1);
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
            const int64_t group = blockIdx.x + static_cast<int64_t>(it / a.nchunks) * gridDim.x;
            const int k = it % a.nchunks;
            // the whole box counts, rows and columns past the matrix included (zero-filled)
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
            tensor_copy_2d(stage0 + static_cast<size_t>(s) * stage_bytes, &wmap, k * kBmChunkBlocks * kBB / 8,
                           static_cast<int>(group * kBmGroupRows), &full[s], wpol);
        };
        // Weights are read-only parameters: one stage streams before the dependency
        // wait, overlapping the preceding kernel's tail. The activation copy goes
        // next and the rest of the ring after it: this CTA's copies are served in
        // issue order, and the fragments (so every stage's use) wait for the
        // activation (Q8_0 14336 x 4096, 8 vectors, chained launches: 13.0 / 12.6 /
        // 13.2 / 13.7 / 14.3 us per launch with 0 / 1 / 2 / 3 / 4 stages ahead of it).
        const int nring = items < STAGES ? items : STAGES;
        issue(0);
        int issued = 1;
        bool ok = true;
        if constexpr (FX) {
            // the consumers' loads of the fp32 activation go out first too: the rest
            // of the ring waits until they are done
            ok = mbar_wait(xready, 0);
        } else {
            pdl_wait();  // the activations may be written by the preceding kernel
            // one bulk copy per vector (whole Q8_0 rows: 16-byte multiples at 16-byte
            // aligned addresses), all on xbar
            mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(a.batch * x_row));
            for (int v = 0; v < a.batch; ++v)
                bulk_copy_g2s(xs + static_cast<size_t>(v) * x_pitch, a.xq + static_cast<int64_t>(v) * a.xq_stride,
                              static_cast<uint32_t>(x_row), xbar, l2_evict_last_policy());
        }
        for (; ok && issued < nring; ++issued) issue(issued);
        for (int it = issued; ok && it < items; ++it) {
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
        if constexpr (!FX) (void)mbar_wait(xbar, 0);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint32_t sel = mma_even_sel(t);
    // the activations may be written, and outputs still read, by the preceding kernel
    pdl_wait();
    bool ok = true;
    if constexpr (FX) {
        // every vector's blocks back to back ([batch][nb] Q8_0 blocks); nb is a
        // multiple of 8, so no quad of blocks straddles two vectors
        quantize_quads_to_smem<kBmWarps>(a.xf, a.batch * (a.nb >> 2), xs, warp, lane);
        bm_consumer_barrier();
        if (tid == 0) mbar_arrive(xready);
    } else {
        // A timed-out wait marks the CTA aborted: the warps skip all further waits
        // and work but keep meeting at the consumer barrier.
        ok = __all_sync(0xffffffffu, mbar_wait(xbar, 0));
        if (!ok) {
            if (lane == 0) atomicOr(a.fault, 1u);
            *abort_flag = 1;
        }
    }
    // Fragments and table from the staged activation: the warp's blocks w, w +
    // kBmWarps, ... (at most kBmMaxBlocks / kBmWarps of them, the plan's limit),
    // lane (g, t) the words t of vector g. Every load is taken before the barrier,
    // every store after it: the fragments overwrite the staged activation.
    constexpr int kU = kBmMaxBlocks / kBmWarps;
    uint32_t r0[kU], r1[kU];
    float dx[kU];
    {
        const uint32_t xv = smem_addr(xs) + static_cast<uint32_t>(g * x_pitch);
        const bool has_v = ok && g < a.batch;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int b = warp + u * kBmWarps;
            r0[u] = 0u;
            r1[u] = 0u;
            dx[u] = 0.0f;
            if (has_v && b < a.nb) bm_load_x<FMT>(xv, b, t, sel, r0[u], r1[u], dx[u]);
        }
    }
    bm_consumer_barrier();  // every load of the staged activation is performed
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int b = warp + u * kBmWarps;  // warp-uniform
        if (b < nb_pad)
            bm_store_block<FMT>(r0[u], r1[u], dx[u], lane, smem_addr(frag) + static_cast<uint32_t>(b * kBmFragBytes),
                                smem_addr(table) + static_cast<uint32_t>(b * kBmTableBytes));
    }
    bm_consumer_barrier();

    const int slab = warp / kBmParts;
    const int part = warp % kBmParts;
    const uint32_t fb0 = smem_addr(frag) + static_cast<uint32_t>(part * kBmWarpBlocks * kBmFragBytes + lane * 16);
    const uint32_t tb0 = smem_addr(table) + static_cast<uint32_t>(part * kBmWarpBlocks * kBmTableBytes + t * 16);
    const uint32_t row_ofs =
        static_cast<uint32_t>((slab * kMmaRows + g) * a.pitch + part * kBmWarpBlocks * kBB);
    int it = 0;
    for (int gi = 0; gi < my_groups; ++gi) {
        const int64_t r0 = (blockIdx.x + static_cast<int64_t>(gi) * gridDim.x) * kBmGroupRows;
        // the warp's blocks 0, 1 of each chunk in acc, blocks 2, 3 in acc2 (two
        // independent fma chains), added at the end of the group
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int k = 0; k < a.nchunks; ++k, ++it) {
            const int s = it % STAGES;
            // A timed-out wait ends this warp's work (every later wait of the
            // other warps is bounded too) and marks the CTA aborted, so no output
            // is stored; the warp keeps meeting the others at the consumer barrier.
            // (The flag is not polled per stage: that vote and shared load on every
            // stage's critical path cost 0.2 us per launch.)
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(it / STAGES) & 1u));
                if (!ok) {
                    if (lane == 0) atomicOr(a.fault, 1u);
                    *abort_flag = 1;
                }
            }
            if (!ok) continue;
            const uint32_t rg = smem_addr(stage0) + static_cast<uint32_t>(s * stage_bytes) + row_ofs;
            const uint32_t rh = rg + static_cast<uint32_t>(8 * a.pitch);
            const uint32_t rgt = rg + static_cast<uint32_t>(4 * t);
            const uint32_t rht = rh + static_cast<uint32_t>(4 * t);
            const uint32_t fb = fb0 + static_cast<uint32_t>(k * kBmChunkBlocks * kBmFragBytes);
            const uint32_t tb = tb0 + static_cast<uint32_t>(k * kBmChunkBlocks * kBmTableBytes);
            BmPair<FMT> p0, p1;
            bm_pair_load<FMT, 0>(p0, rg, rgt, rh, rht, fb, tb, sel);
            bm_pair_load<FMT, 1>(p1, rg, rgt, rh, rht, fb, tb, sel);
            // The warp's bytes of the stage are in registers now: the stage is
            // released before the arithmetic (the arrival's release semantics
            // order the warp's shared loads before it, and the producer fences
            // the async proxy before it copies into the stage again), so it is
            // held for the loads only and the ring keeps more copies in flight.
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            bm_pair_compute<FMT>(p0, acc);
            bm_pair_compute<FMT>(p1, acc2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = __fadd_rn(acc[q], acc2[q]);
        // the slab's 8 partial sums, added in part order: thread o < 256 takes
        // output (slab o / 128, vector (o % 128) / 16, row o % 16)
        const uint32_t rb = smem_addr(red) + static_cast<uint32_t>((a.red_bufs == 2 ? (gi & 1) : 0) * kBmRedBytes);
        if (a.red_bufs == 1 && gi > 0) bm_consumer_barrier();  // the previous group's sums are read
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(rb + static_cast<uint32_t>(warp * 512 + lane * 16)),
                     "f"(acc[0]), "f"(acc[1]), "f"(acc[2]), "f"(acc[3])
                     : "memory");
        bm_consumer_barrier();
        if (tid < kBmSlabs * kMmaRows * 8 && !*abort_flag) {
            const int j = tid >> 7;
            const int v = (tid >> 4) & 7;
            const int r = tid & 15;
            // lane (r % 8) * 4 + v / 2 holds (row r, vector v) at element (r / 8) * 2 + v % 2
            const uint32_t e = static_cast<uint32_t>((((r & 7) * 4 + (v >> 1)) * 4 + (r >> 3) * 2 + (v & 1)) * 4);
            float sum = 0.0f;
#pragma unroll
            for (int p = 0; p < kBmParts; ++p)
                sum = __fadd_rn(sum, __uint_as_float(lds32(rb + static_cast<uint32_t>((j * kBmParts + p) * 512) + e)));
            const int64_t row = r0 + j * kMmaRows + r;
            if (v < a.batch && row < a.rows) a.y[static_cast<int64_t>(v) * a.y_stride + row] = sum;
        }
    }
}

template <int FMT, int STAGES, bool FX>
struct BmmaInst {
    static constexpr auto kKernel = &dmmv_bmma_kernel<FMT, STAGES, FX>;
    // one CTA per SM (at most one per 32-row group)
    static cudaError_t launch(const BmmaArgs &a, const CUtensorMap &wmap, int smem_bytes, cudaStream_t st, bool pdl) {
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
        const int64_t ngroups = (a.rows + kBmGroupRows - 1) / kBmGroupRows;
        const int64_t ctas = ngroups < sms ? ngroups : sms;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
        cfg.blockDim = dim3((kBmWarps + 1) * 32, 1, 1);
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

}  // namespace zdmmv
