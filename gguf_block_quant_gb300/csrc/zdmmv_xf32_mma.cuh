// zdmmv_xf32_mma.cuh -- the decode DMMV with the activation taken as fp32 values,
// on the fp16 tensor cores (GGUF layout), for sm_103a.
//
// y[r] = sum_b d_w[r,b] * sum_i v[r,b,i] * x[b,i], x as given (the ZINC_RT
// slice's f32 input vector: "The first ZINC_RT model slices that actually
// count", kernel ABI). The scalar kernel (zdmmv_xf32.cuh) spends a byte permute,
// a subtraction and an fma on every weight and is bound by instruction issue.
// Here the weight codes (Q8_0: -128..127; Q4_0: q - 8) become exact fp16 values,
// two per instruction pair, and mma.sync.m16n8k16 multiplies 16 rows x 16 codes
// by the activation at once:
//  * each 32-value block of x is scaled by a power of two 2^s (its largest
//    magnitude lands in [2^14, 2^15)) and split into three fp16 parts,
//    h1 = fp16(u), h2 = fp16(u - h1), h3 = fp16(u - h1 - h2) for u = x * 2^s;
//    their sum is u exactly (elements below 2^-15 of the block's largest lose
//    bits under 2^-39 of it), and the parts are the MMA's columns 0..2;
//  * fp16 x fp16 products are exact in fp32, the block's two MMAs accumulate in
//    fp32, and each part's block result is scaled by d_w * 2^-s and accumulated
//    in fp32 (acc = fma(coef, D, acc)); y adds the three parts.
// The order of the fp32 sums differs from the scalar kernel, so the results
// agree with it within the fp32 tolerance, not bit for bit.
//
// The weights stream as described in zdmmv_mma.cuh: a producer warp issues one
// 2D tensor copy per stage (a group of 16-row slabs, one per consumer warp, by a
// chunk of blocks) whose shared-memory pitch is 4 mod 8 words, so the fragment
// loads of the 8 rows of a lane quad hit distinct banks; the lane loads the
// aligned words of each GGUF block pair (XmRow, at immediate offsets, 8 blocks per
// stage, the pairs unrolled) and the k-slot of each code is chosen to match the
// word it arrives in; the activation fragments use the same order.
#pragma once

#include <cuda_fp16.h>

#include "zdmmv_mma.cuh"

namespace zdmmv {

struct Xf32MmaArgs {
    const uint8_t *w;    // GGUF rows
    const float *xf;     // fp32 activation of slot 0 (blockIdx.y = slot)
    float *y;            // output of slot 0
    uint32_t *fault;     // device fault word
    int64_t rows;
    int64_t xf_stride;   // floats between slots' activations
    int64_t y_stride;    // floats between slots' outputs
    int32_t nb;          // blocks per row
    int32_t cb;          // blocks per row in one stage
    int32_t nchunks;     // stages per row group
    int32_t pitch;       // shared-memory bytes per staged row
};

// per block: 12 lanes x 16 bytes of fp16 parts, 2^-s at byte 192, 16 zero bytes at 208
constexpr int kXmFragBytes = 256;
constexpr int kXmZeroOfs = 208;  // the zero slot (lanes without a part)
// Blocks per row in one stage (a chunk); 8 blocks = 144 (Q4_0) or 272 (Q8_0)
// bytes, 4 mod 8 words, so the chunk needs no padding for conflict-free loads.
constexpr int kXmChunkBlocks = 8;

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C (f32)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// The 8 codes of one Q4_0 quant word (bytes B0..B3) as exact fp16 pairs:
// lo02 = (lo(B0) - 8, lo(B2) - 8), lo13, hi02 = (hi(B0) - 8, hi(B2) - 8), hi13.
// A nibble n in the low bits of 0x6400 reads as 1024 + n (the fp16 unit there is
// 1); in bits 4..7 as 1024 + 16 n, which (x / 16) - 72 brings to n - 8.
struct Q4Halves {
    uint32_t lo02, lo13, hi02, hi13;
};
__device__ __forceinline__ Q4Halves q4_halves(uint32_t w) {
    constexpr uint32_t kMagic = 0x64006400u;      // fp16 1024, both halves
    constexpr uint32_t k1032 = 0x64086408u;       // fp16 1032 = 1024 + 8
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16
    constexpr uint32_t kMinus72 = 0xD480D480u;    // fp16 -72 = -(1024 / 16 + 8)
    const uint32_t s = w >> 8;
    Q4Halves h;
    h.lo02 = h2_sub((w & 0x000F000Fu) | kMagic, k1032);
    h.lo13 = h2_sub((s & 0x000F000Fu) | kMagic, k1032);
    h.hi02 = h2_fma((w & 0x00F000F0u) | kMagic, kSixteenth, kMinus72);
    h.hi13 = h2_fma((s & 0x00F000F0u) | kMagic, kSixteenth, kMinus72);
    return h;
}

// The 4 codes c0..c3 of one Q8_0 word as exact fp16 pairs (c0, c2) and (c1, c3):
// the offset byte c + 128 under 0x64 reads as 1024 + c + 128.
__device__ __forceinline__ void q8_halves(uint32_t w, uint32_t &p02, uint32_t &p13) {
    constexpr uint32_t k1152 = 0x64806480u;  // fp16 1152 = 1024 + 128
    const uint32_t u = w ^ 0x80808080u;
    p02 = h2_sub(__byte_perm(u, 0x64646464u, 0x4240u), k1152);
    p13 = h2_sub(__byte_perm(u, 0x64646464u, 0x4341u), k1152);
}

// A fragments of one block for rows g and g + 8 (the lane's quant words, XmRow):
// a0 for the first MMA (codes of the block's k-slots 0..15), a1 for the
// second. Fragment register order {row g, row g + 8} x {k-pair (2t, 2t+1),
// k-pair (2t+8, 2t+9)}.
template <int FMT> struct XmFrags;
template <> struct XmFrags<kFmtQ4> {
    __device__ __forceinline__ static void make(uint32_t wg, uint32_t wh, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
        const Q4Halves g = q4_halves(wg), h = q4_halves(wh);
        a0[0] = g.lo02;
        a0[1] = h.lo02;
        a0[2] = g.lo13;
        a0[3] = h.lo13;
        a1[0] = g.hi02;
        a1[1] = h.hi02;
        a1[2] = g.hi13;
        a1[3] = h.hi13;
    }
};
template <> struct XmFrags<kFmtQ8> {
    __device__ __forceinline__ static void make(uint32_t ag, uint32_t bg, uint32_t ah, uint32_t bh, uint32_t (&a0)[4],
                                                uint32_t (&a1)[4]) {
        q8_halves(ag, a0[0], a0[2]);
        q8_halves(ah, a0[1], a0[3]);
        q8_halves(bg, a1[0], a1[2]);
        q8_halves(bh, a1[1], a1[3]);
    }
};

// The element (0..31) of a block that lane t's fragment slot k (0..7) faces:
// slots {MMA 0: k-pair (2t, 2t+1) low, high, k-pair (2t+8, 2t+9) low, high;
// MMA 1: the same}. Byte c of a quant word lands in slot order c0, c2, c1, c3
// (the fp16 pairs (0, 2) and (1, 3)). Q4_0: the lane's word holds quant bytes
// j_c = 4t + c (odd block) or (4t + 2 + c) mod 16 (even block), low nibbles =
// elements j_c (MMA 0), high nibbles = j_c + 16 (MMA 1). Q8_0: the words hold
// codes 4t + c and 16 + 4t + c (odd block), 2 + 4t + c and 18 + 4t + c (even
// block; the last lane of a quad 30, 31, 0, 1 for the second).
template <int FMT>
__device__ __forceinline__ int xm_element(bool odd, int t, int k) {
    const int c = ((k & 1) << 1) | ((k >> 1) & 1);
    if constexpr (FMT == kFmtQ4) {
        const int j = odd ? 4 * t + c : (4 * t + 2 + c) & 15;
        return k >= 4 ? j + 16 : j;
    } else {
        if (k < 4) return odd ? 4 * t + c : 2 + 4 * t + c;
        if (odd) return 16 + 4 * t + c;
        return t < 3 ? 18 + 4 * t + c : (c < 2 ? 30 + c : c - 2);
    }
}

// Activation fragments of block b (one warp; v = element `lane` of the block):
// the block's scale 2^s from its largest magnitude, the three fp16 parts of every element, and for lane (g, t),
// g < 3, part g of the 8 elements its slots face (16 bytes at lane * 16); 2^-s at
// byte 192; zeros at kXmZeroOfs.
template <int FMT>
__device__ __forceinline__ void xm_build_block(float v, int b, int lane, uint32_t frag) {
    // for non-negative floats the bit patterns order like the values
    const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
    int s = 0;
    if (m != 0.0f) {
        const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu) - 127;  // 2^e <= m < 2^(e+1)
        s = 14 - e;
        s = s > 126 ? 126 : (s < -126 ? -126 : s);
    }
    const float u = __fmul_rn(v, __int_as_float((s + 127) << 23));
    const __half h1 = __float2half_rn(u);
    const float r1 = __fsub_rn(u, __half2float(h1));
    const __half h2 = __float2half_rn(r1);
    const float r2 = __fsub_rn(r1, __half2float(h2));
    const __half h3 = __float2half_rn(r2);
    const uint32_t p12 = static_cast<uint32_t>(__half_as_ushort(h1)) |
                         (static_cast<uint32_t>(__half_as_ushort(h2)) << 16);
    const uint32_t p3 = __half_as_ushort(h3);
    const int g = lane >> 2;
    const int t = lane & 3;
    const bool odd = (b & 1) != 0;
    uint32_t f[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int src = xm_element<FMT>(odd, t, k);
        const uint32_t a = __shfl_sync(0xffffffffu, p12, src);
        const uint32_t c = __shfl_sync(0xffffffffu, p3, src);
        const uint32_t part = g == 0 ? (a & 0xffffu) : (g == 1 ? (a >> 16) : (c & 0xffffu));
        f[k >> 1] |= part << (16 * (k & 1));
    }
    if (g < 3)
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(frag + static_cast<uint32_t>(lane * 16)),
                     "r"(f[0]), "r"(f[1]), "r"(f[2]), "r"(f[3])
                     : "memory");
    if (lane == 0)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(frag + 192u), "f"(__int_as_float((127 - s) << 23)) : "memory");
    if (lane == 1)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(frag + static_cast<uint32_t>(kXmZeroOfs)),
                     "r"(0u)
                     : "memory");
}

// One block's two MMAs and the fp32 update: coef_g, coef_h = d_w * 2^-s of rows
// g and g + 8.
__device__ __forceinline__ void xm_block(const uint32_t (&a0)[4], const uint32_t (&a1)[4], const uint4 &f,
                                         float coef_g, float coef_h, float (&acc)[4]) {
    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float d[4];
    mma_16816(d, a0, f.x, f.y, zero);
    mma_16816(d, a1, f.z, f.w, d);
    acc[0] = __fmaf_rn(coef_g, d[0], acc[0]);
    acc[1] = __fmaf_rn(coef_g, d[1], acc[1]);
    acc[2] = __fmaf_rn(coef_h, d[2], acc[2]);
    acc[3] = __fmaf_rn(coef_h, d[3], acc[3]);
}

// Shared-memory loads at a compile-time offset from a base address (the offset
// goes into the instruction, no address arithmetic per load). Volatile like
// lds32, so they are never hoisted above the wait that makes the data valid.
template <int OFS>
__device__ __forceinline__ uint32_t ldsi(uint32_t base) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(base), "n"(OFS));
    return v;
}
template <int OFS>
__device__ __forceinline__ uint4 ldsi128(uint32_t base) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(base), "n"(OFS));
    return v;
}


// One block pair P (blocks 2P, 2P + 1 of the chunk) of one row of a stage, at
// immediate offsets from r = the staged row and rt = r + 4t: both blocks' scales
// and lane t's aligned code words. Q8_0: words (k-slots of MMA 0, of MMA 1) of the
// even block, codes 2 + 4t.. and 18 + 4t.. (ea, eb; the last lane's eb completed
// from the pair's first word) and of the odd block, codes 4t.. and 16 + 4t.. (oa,
// ob). Q4_0: one word of quant bytes per block (ea, oa), its low nibbles for MMA
// 0 and its high nibbles for MMA 1.
template <int FMT> struct XmRow;
template <> struct XmRow<kFmtQ4> {
    uint32_t ea, oa;
    float d0, d1;
    template <int P>
    __device__ __forceinline__ void load(uint32_t r, uint32_t rt, uint32_t sel) {
        constexpr int kP = 36 * P;
        const uint32_t e0 = ldsi<kP>(r);       // d0 | quant bytes 0, 1
        const uint32_t e4 = ldsi<kP + 16>(r);  // quant bytes 14, 15 | d1
        ea = __byte_perm(ldsi<kP + 4>(rt), e0, sel);
        oa = ldsi<kP + 20>(rt);
        d0 = half_lo(e0);
        d1 = half_hi(e4);
    }
};
template <> struct XmRow<kFmtQ8> {
    uint32_t ea, eb, oa, ob;
    float d0, d1;
    template <int P>
    __device__ __forceinline__ void load(uint32_t r, uint32_t rt, uint32_t sel) {
        constexpr int kP = 68 * P;
        const uint32_t e0 = ldsi<kP>(r);       // d0 | codes 0, 1
        const uint32_t e8 = ldsi<kP + 32>(r);  // codes 30, 31 | d1
        ea = ldsi<kP + 4>(rt);
        eb = __byte_perm(ldsi<kP + 20>(rt), e0, sel);
        oa = ldsi<kP + 36>(rt);
        ob = ldsi<kP + 52>(rt);
        d0 = half_lo(e0);
        d1 = half_hi(e8);
    }
};

// Pair P of a stage for this lane: rows g (rg, rgt) and g + 8 (rh, rht); fb: the
// chunk's fragment base for this lane (its 16-byte slot, or the zero slot), sb:
// the chunk's first scale. Two blocks, four MMAs, eight fp32 updates.
template <int FMT, int P>
__device__ __forceinline__ void xm_pair(uint32_t rg, uint32_t rgt, uint32_t rh, uint32_t rht, uint32_t fb,
                                        uint32_t sb, uint32_t sel, float (&acc)[4]) {
    constexpr int kF = 2 * P * kXmFragBytes;
    XmRow<FMT> wg, wh;
    wg.template load<P>(rg, rgt, sel);
    wh.template load<P>(rh, rht, sel);
    const uint4 f0 = ldsi128<kF>(fb);
    const uint4 f1 = ldsi128<kF + kXmFragBytes>(fb);
    const float inv0 = __uint_as_float(ldsi<kF>(sb));
    const float inv1 = __uint_as_float(ldsi<kF + kXmFragBytes>(sb));
    uint32_t a0[4], a1[4];
    if constexpr (FMT == kFmtQ4) {
        XmFrags<kFmtQ4>::make(wg.ea, wh.ea, a0, a1);
        xm_block(a0, a1, f0, __fmul_rn(wg.d0, inv0), __fmul_rn(wh.d0, inv0), acc);
        XmFrags<kFmtQ4>::make(wg.oa, wh.oa, a0, a1);
        xm_block(a0, a1, f1, __fmul_rn(wg.d1, inv1), __fmul_rn(wh.d1, inv1), acc);
    } else {
        XmFrags<kFmtQ8>::make(wg.ea, wg.eb, wh.ea, wh.eb, a0, a1);
        xm_block(a0, a1, f0, __fmul_rn(wg.d0, inv0), __fmul_rn(wh.d0, inv0), acc);
        XmFrags<kFmtQ8>::make(wg.oa, wg.ob, wh.oa, wh.ob, a0, a1);
        xm_block(a0, a1, f1, __fmul_rn(wg.d1, inv1), __fmul_rn(wh.d1, inv1), acc);
    }
}

// NW consumer warps + 1 producer warp. A stage holds NW x 16 rows (a row group)
// by a chunk of a.cb blocks; warp w takes rows 16w .. 16w + 15 of every stage,
// so each warp owns whole rows and needs no combine with the others. CTA (c,
// slot) takes the slot's row groups c, c + gridDim.x, ..., each in a.nchunks
// stages. wmap: the weight rows as a 2D tensor of 8-byte elements, box
// {a.pitch / 8, NW * 16}.
template <int FMT, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32, 2) dmmv_xf32_mma_kernel(const Xf32MmaArgs a,
                                                                         const __grid_constant__ CUtensorMap wmap) {
    constexpr int kBB = Fmt<FMT>::kBlockBytes;
    constexpr int kConsumers = NW * 32;
    constexpr int kGroupRows = NW * kMmaRows;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xready = empty + STAGES;  // the consumers have built the activation fragments
    uint8_t *frag = smem + kBarrierBytes;
    uint8_t *stage0 = frag + static_cast<size_t>(a.nb) * kXmFragBytes;
    const int stage_bytes = kGroupRows * a.pitch;

    const int tid = threadIdx.x;
    const int slot = blockIdx.y;
    const float *x = a.xf + slot * a.xf_stride;
    float *y = a.y + slot * a.y_stride;
    const int64_t ngroups = (a.rows + kGroupRows - 1) / kGroupRows;
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
            mbar_init(&empty[s], NW);
        }
        mbar_init(xready, 1);
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
            tensor_copy_2d(stage0 + static_cast<size_t>(s) * stage_bytes, &wmap, k * a.cb * kBB / 8,
                           static_cast<int>(group * kGroupRows), &full[s], wpol);
        };
        // Weights are read-only parameters: one stage streams before the
        // consumers' activation loads, the rest of the ring once the fragments are
        // built (loads issued behind the whole ring of this CTA's weight copies
        // would wait for all of them).
        const int nring = items < STAGES ? items : STAGES;
        issue(0);
        int issued = 1;
        bool ok = mbar_wait(xready, 0);
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
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint32_t sel = mma_even_sel(t);
    pdl_wait();  // the activation may be written, and y still read, by the preceding kernel
    // the warp's blocks w, w + NW, ...: 8 at a time, their loads all in flight first
    for (int b0 = warp; b0 < a.nb; b0 += 8 * NW) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int b = b0 + u * NW;
            v[u] = b < a.nb ? x[static_cast<int64_t>(b) * kQK + lane] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int b = b0 + u * NW;  // warp-uniform
            if (b < a.nb) xm_build_block<FMT>(v[u], b, lane, smem_addr(frag) + static_cast<uint32_t>(b * kXmFragBytes));
        }
    }
    mma_consumer_barrier<NW>();
    if (tid == 0) mbar_arrive(xready);

    // lanes of quads 0..2 hold activation parts 0..2; the others load 16 zero bytes
    const uint32_t frag_l = smem_addr(frag) + static_cast<uint32_t>(g < 3 ? lane * 16 : kXmZeroOfs);
    const uint32_t scale_a = smem_addr(frag) + 192u;
    const uint32_t row_ofs = static_cast<uint32_t>((warp * kMmaRows + g) * a.pitch);
    int it = 0;
    for (int gi = 0; gi < my_groups; ++gi) {
        const int64_t r0 = (blockIdx.x + static_cast<int64_t>(gi) * gridDim.x) * kGroupRows + warp * kMmaRows;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int k = 0; k < a.nchunks; ++k, ++it) {
            const int s = it % STAGES;
            // a timed-out wait leaves the kernel: nothing else in this warp waits after it
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(it / STAGES) & 1u))) {
                if (lane == 0) atomicOr(a.fault, 1u);
                return;
            }
            const uint32_t rg = smem_addr(stage0) + static_cast<uint32_t>(s * stage_bytes) + row_ofs;
            const uint32_t rh = rg + static_cast<uint32_t>(8 * a.pitch);
            const uint32_t rgt = rg + static_cast<uint32_t>(4 * t);
            const uint32_t rht = rh + static_cast<uint32_t>(4 * t);
            const uint32_t kf = static_cast<uint32_t>(k * kXmChunkBlocks * kXmFragBytes);
            const uint32_t fb = frag_l + kf;
            const uint32_t sb = scale_a + kf;
            xm_pair<FMT, 0>(rg, rgt, rh, rht, fb, sb, sel, acc);
            xm_pair<FMT, 1>(rg, rgt, rh, rht, fb, sb, sel, acc);
            xm_pair<FMT, 2>(rg, rgt, rh, rht, fb, sb, sel, acc);
            xm_pair<FMT, 3>(rg, rgt, rh, rht, fb, sb, sel, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // rows g and g + 8 of the warp's slab: parts 0, 1 sit in lane quad member 0
        // (acc[0], acc[1]; acc[2], acc[3] for row g + 8), part 2 in member 1
        const float p2g = __shfl_down_sync(0xffffffffu, acc[0], 1);
        const float p2h = __shfl_down_sync(0xffffffffu, acc[2], 1);
        if (t == 0) {
            if (r0 + g < a.rows) y[r0 + g] = __fadd_rn(__fadd_rn(acc[0], acc[1]), p2g);
            if (r0 + g + 8 < a.rows) y[r0 + g + 8] = __fadd_rn(__fadd_rn(acc[2], acc[3]), p2h);
        }
    }
}

template <int FMT, int NW, int STAGES>
struct Xf32MmaInst {
    static constexpr auto kKernel = &dmmv_xf32_mma_kernel<FMT, NW, STAGES>;
    // one wave of the CTAs that fit, split over the slots
    static cudaError_t launch(const Xf32MmaArgs &a, const CUtensorMap &wmap, int smem_bytes, int slots,
                              cudaStream_t st, bool pdl) {
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
        int per_sm = 0;
        const uint64_t c = occ_cache[dev].load(std::memory_order_relaxed);
        if (c != 0 && static_cast<int>(c >> 32) == smem_bytes) {
            per_sm = static_cast<int>(c & 0xffffffffu);
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kKernel, (NW + 1) * 32,
                                                              static_cast<size_t>(smem_bytes));
            if (e != cudaSuccess) return e;
            per_sm = per_sm > 0 ? per_sm : 1;
            occ_cache[dev].store((static_cast<uint64_t>(smem_bytes) << 32) | static_cast<uint32_t>(per_sm),
                                 std::memory_order_relaxed);
        }
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t ngroups = (a.rows + NW * kMmaRows - 1) / (NW * kMmaRows);
        int64_t ctas = static_cast<int64_t>(sms) * per_sm / slots;
        if (ctas < 1) ctas = 1;
        if (ctas > ngroups) ctas = ngroups;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), static_cast<unsigned>(slots), 1);
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

}  // namespace zdmmv
