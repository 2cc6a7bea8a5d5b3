// zdmmv_device.cuh -- device building blocks of the GB300 (sm_103a) decode DMMV.
//
// * inline-PTX wrappers for mbarriers, the bulk (TMA) global->shared copy and
//   the mixed-signedness packed int8x4 dot product;
// * the block arithmetic: for every (format, layout) pair a "Pair" type that
//   holds one lane's slice of the Q8_0 activation in registers and turns the
//   weight words of two consecutive blocks into the two int32 block sums and
//   their fp32 contribution.
//
// Block arithmetic (per 32-element block, int32, exact):
//   Q8_0:  s = sum_i qw_i * qx_i                        (8 x dp4a)
//   Q4_0:  s = sum_i (q_i - 8) * qx_i
//            = sum_{j<16} lo(qs_j)*qx_j + sum_{j<16} hi(qs_j)*qx_{j+16} - 8*sum_i qx_i
// and per block the fp32 update acc = fma(float(s), d_w*d_x, acc) where
// d_w*d_x of two fp16 values is exact in fp32 and |s| <= 32*128*127 < 2^24 is
// exact as a float. The int8x4 dot is the operation the pages build every
// quantized matvec on ("Bringing ZINC to NVIDIA: a CUDA backend", section "The
// reassuring result: ZINC's matmuls are __dp4a, not tensor cores"); the -8
// offset of Q4_0 is the Q4 unpack in the habr ZINC article, "Что такое DMMV".
//
// GGUF array-of-blocks rows put a block every 34 (Q8_0) or 18 (Q4_0) bytes, so
// half the blocks start 2 bytes off a 4-byte boundary. Instead of realigning the
// weight words (a byte permute per word), a lane owns PAIRS of blocks (68 or 36
// bytes, always 4-byte aligned when the row is) and holds its activation words
// pre-shifted to the weight words' alignment, with zero bytes facing the fp16
// scale bytes: the dp4a of a scale byte with a zero contributes nothing, so the
// unaligned block needs no permutes at all.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace zdmmv {

constexpr int kQK = 32;
constexpr int kFmtQ4 = 2;
constexpr int kFmtQ8 = 8;
constexpr int kLayoutGguf = 0;
constexpr int kLayoutRepacked = 1;

template <int FMT> struct Fmt;
template <> struct Fmt<kFmtQ8> { static constexpr int kBlockBytes = 34; static constexpr int kQuantBytes = 32; };
template <> struct Fmt<kFmtQ4> { static constexpr int kBlockBytes = 18; static constexpr int kQuantBytes = 16; };

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Explicit shared-memory loads (addresses from smem_addr): the compiler cannot
// always prove that a pointer handed through the block-arithmetic helpers points
// into shared memory, and a generic load takes the slower global-memory path.
// They are volatile so that they are never hoisted above the barrier wait that
// makes the data valid.
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Lane l of a row group of LPR lanes owns block pairs l, l + LPR, ... (pair j of
// the lane is l + j*LPR): in every layout consecutive lanes read consecutive pair
// slots, and both layouts sum a row's pairs in the same order.
template <int LPR>
__device__ __forceinline__ int owned_pair(int l, int j) { return l + j * LPR; }

// Sum over the G lanes of a row group (G = 8, 16 or 32; groups are aligned lane
// ranges of a warp) of N values per lane (N a power of two, N <= G), scattered:
// lane l of the group ends with the group sum of value l / (G / N). The values
// are exchanged from the highest lane bit down, halving the set at each of the
// first log2(N) steps; every value is combined over the same pairs of lanes, in
// the same order of bits, as the plain xor tree (acc += shfl_xor(acc, o) for
// o = G/2 .. 1), so each sum is bitwise the one that tree gives.
template <int G, int N>
__device__ __forceinline__ float group_reduce_scatter(const float (&v)[N], int l) {
    static_assert(N >= 1 && N <= G && (N & (N - 1)) == 0, "N a power of two <= G");
    float cur[N];
#pragma unroll
    for (int k = 0; k < N; ++k) cur[k] = v[k];
    int bit = G / 2;
#pragma unroll
    for (int width = N; width > 1; width >>= 1, bit >>= 1) {
        const bool upper = (l & bit) != 0;
#pragma unroll
        for (int k = 0; k < width / 2; ++k) {
            const float send = upper ? cur[k] : cur[width / 2 + k];
            const float keep = upper ? cur[width / 2 + k] : cur[k];
            cur[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = cur[0];
#pragma unroll
    for (int o = G / (2 * N); o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// unsigned bytes of a times signed bytes of b, accumulated into c (int32)
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every wait in this library is bounded: after this long (or this many polls,
// whichever comes first) the waiter gives up, the kernel records
// ZDMMV_FAULT_WAIT_TIMEOUT and returns instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr uint32_t kWaitMaxPolls = 1u << 26;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t polls = 0; !mbar_try_wait(bar, parity); ++polls) {
        if (polls >= kWaitMaxPolls || global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`. dst, src 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// fp16 bits held in the low / high half of a 32-bit word, as float (exact)
__device__ __forceinline__ float half_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// bytes 2,3 of a followed by bytes 0,1 of b: a 4-byte window shifted by 2 bytes
__device__ __forceinline__ uint32_t shift2(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5432); }

constexpr uint32_t kLoNib = 0x0f0f0f0fu;
constexpr uint32_t kHiNib = 0xf0f0f0f0u;
constexpr uint32_t kOnes = 0x01010101u;

// Q8_0 quantization of one 32-element block held one element per lane of a full
// warp: amax = max|x_i|; d = amax/127 (IEEE division); id = d ? 1/d : 0 (IEEE
// reciprocal); q_i = round(x_i*id) (fp32 product, ties away from zero); the scale
// is stored as fp16(d), round to nearest even. Returns this lane's code and the
// scale bits. The same function serves the stand-alone quantizer and the fused
// DMMV prologue, so both produce identical bytes.
__device__ __forceinline__ int quantize_q8_0_lane(float v, unsigned short &d_bits) {
    // for non-negative floats the bit patterns order like the values
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    d_bits = __half_as_ushort(__float2half_rn(d));
    return static_cast<int>(roundf(__fmul_rn(v, id)));
}

// The same quantizer with four blocks per warp: lanes 8k..8k+7 hold block k's
// elements (4 per lane, lane 8k+j has elements 4j..4j+3). The block maximum is an
// exact max, reduced over the 8 lanes, and d, id and the codes use exactly the
// operations of quantize_q8_0_lane, so the bytes are identical. Returns the four
// codes packed little-endian.
__device__ __forceinline__ uint32_t quantize_q8_0_quad(float4 v, unsigned short &d_bits) {
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    const float d = m / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    d_bits = __half_as_ushort(__float2half_rn(d));
    const uint32_t q0 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.x, id)))));
    const uint32_t q1 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.y, id)))));
    const uint32_t q2 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.z, id)))));
    const uint32_t q3 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.w, id)))));
    return q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
}

// One round of quantize_quads_to_smem: the loads of kRound quads of the warp
// (quads q0, q0 + kWarps, ...; zeros past nquads, no access).
template <int kWarps, int kRound>
__device__ __forceinline__ void quantize_round_load(const float *xf, int nquads, int q0, int sub, int j,
                                                    float4 (&v)[kRound]) {
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
        const int qd = q0 + u * kWarps;
        v[u] = qd < nquads ? *reinterpret_cast<const float4 *>(xf + static_cast<int64_t>(4 * qd + sub) * kQK + 4 * j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// The rest of a round: block maxima, scales and codes, stored into xs.
template <int kWarps, int kRound>
__device__ __forceinline__ void quantize_round_store(const float4 (&v)[kRound], int nquads, int q0, uint8_t *xs,
                                                     int lane, int sub, int j) {
    float m[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u)
        m[u] = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
        for (int u = 0; u < kRound; ++u) m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], o));
    }
    // the operations of quantize_q8_0_lane (IEEE division and reciprocal),
    // once per block: lane j of the 8 sharing a block takes round j's block
    // and the results are broadcast to the other 7
    static_assert(kRound == 8, "one round per lane of a block's 8 lanes");
    float mj = m[0];
#pragma unroll
    for (int u = 1; u < kRound; ++u) mj = j == u ? m[u] : mj;
    const float dj = __fdiv_rn(mj, 127.0f);
    const float idj = dj != 0.0f ? __frcp_rn(dj) : 0.0f;
    const uint32_t dbj = __half_as_ushort(__float2half_rn(dj));
    float id[kRound];
    unsigned short db[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
        const int src = (lane & ~7) | u;
        id[u] = __shfl_sync(0xffffffffu, idj, src);
        db[u] = static_cast<unsigned short>(__shfl_sync(0xffffffffu, dbj, src));
    }
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
        const int qd = q0 + u * kWarps;
        if (qd < nquads) {  // warp-uniform
            const uint32_t c0 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v[u].x, id[u])))));
            const uint32_t c1 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v[u].y, id[u])))));
            const uint32_t c2 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v[u].z, id[u])))));
            const uint32_t c3 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v[u].w, id[u])))));
            uint8_t *blk = xs + 34 * (4 * qd + sub);
            uint16_t *dst = reinterpret_cast<uint16_t *>(blk + 2 + 4 * j);  // 2-byte aligned
            dst[0] = static_cast<uint16_t>(c0 | (c1 << 8));
            dst[1] = static_cast<uint16_t>(c2 | (c3 << 8));
            if (j == 0) *reinterpret_cast<unsigned short *>(blk) = db[u];
        }
    }
}

// Quantize 4 * nquads consecutive Q8_0 blocks of the fp32 values at xf into
// shared memory at xs (34 bytes per block), with the stand-alone quantizer's
// arithmetic (quantize_q8_0_lane: fp32 amax, IEEE d = amax / 127 and 1 / d,
// codes round(x * id) with ties away from zero, fp16 scale RNE), so the bytes are
// that quantizer's. The kWarps warps of the calling group (this one is `warp`)
// each take four blocks per iteration (16-byte loads, 8 lanes per block),
// kRound iterations at a time in phases (all loads, all block maxima, all
// scales, all codes) so independent blocks overlap. kAhead: each round's loads
// are issued before the previous round is quantized, so a warp with several
// rounds (batches of vectors) does not wait a whole load latency per round; it
// costs kRound float4 registers. The vector-split kernel turns it on (Q8_0
// 14336 x 4096, 2 / 4 vectors: 12.66 -> 12.32 / 15.69 -> 15.10 us per fused
// launch); the tensor-core batched kernel measured slower with it (8 vectors:
// 16.07 -> 16.38 us) and leaves it off, as do the single-vector callers (one
// round per warp). The caller synchronizes the group before the blocks are read.
template <int kWarps, int kRound = 8, bool kAhead = false>
__device__ __forceinline__ void quantize_quads_to_smem(const float *xf, int nquads, uint8_t *xs, int warp,
                                                       int lane) {
    const int sub = lane >> 3;  // block within the quad
    const int j = lane & 7;     // 4-element group within the block
    constexpr int kStep = kWarps * kRound;
    if constexpr (kAhead) {
        float4 v[kRound], next[kRound];
        quantize_round_load<kWarps, kRound>(xf, nquads, warp, sub, j, v);
        for (int q0 = warp; q0 < nquads; q0 += kStep) {
            quantize_round_load<kWarps, kRound>(xf, nquads, q0 + kStep, sub, j, next);
            quantize_round_store<kWarps, kRound>(v, nquads, q0, xs, lane, sub, j);
#pragma unroll
            for (int u = 0; u < kRound; ++u) v[u] = next[u];
        }
    } else {
        for (int q0 = warp; q0 < nquads; q0 += kStep) {
            float4 v[kRound];
            quantize_round_load<kWarps, kRound>(xf, nquads, q0, sub, j, v);
            quantize_round_store<kWarps, kRound>(v, nquads, q0, xs, lane, sub, j);
        }
    }
}

// Sum of the 32 int8 codes of an activation block, times -8 (the Q4_0 offset
// term), from its eight aligned code words.
__device__ __forceinline__ int q4_offset_term(const uint32_t (&xw)[8]) {
    int s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) s = dp4a_ss(xw[k], kOnes, s);
    return -8 * s;
}

// Load the 17 words of the activation pair p (blocks 2p, 2p+1; 68 bytes at a
// 4-byte aligned offset) from Q8_0 activation blocks at `xq`.
__device__ __forceinline__ void load_x_pair_words(const uint8_t *xq, int p, uint32_t (&v)[17]) {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + 68 * p);
#pragma unroll
    for (int k = 0; k < 17; ++k) v[k] = src[k];
}
// The same from activation blocks staged in shared memory at address xs.
__device__ __forceinline__ void load_x_pair_words_smem(uint32_t xs, int p, uint32_t (&v)[17]) {
#pragma unroll
    for (int k = 0; k < 17; ++k) v[k] = lds32(xs + 68 * p + 4 * k);
}

// Aligned code words of the two activation blocks of a pair:
// block A's 32 codes start at byte 2, block B's at byte 36 of the pair.
__device__ __forceinline__ void x_aligned_words(const uint32_t (&v)[17], uint32_t (&xa)[8], uint32_t (&xb)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        xa[k] = shift2(v[k], v[k + 1]);
        xb[k] = v[9 + k];
    }
}

// -------------------------------------------------------------- Pair types
// Pair<FMT, LAYOUT>: one lane's registers for one pair of blocks and the update
//   acc = fma(float(sA), dwA*dxA, acc); acc = fma(float(sB), dwB*dxB, acc)
// in that order. `sums()` returns the two int32 block sums (debug path).
template <int FMT, int LAYOUT> struct Pair;

// Q8_0, GGUF layout. Weight pair words w[0..16] (68 bytes):
//   w0 = [dA dA a0 a1], w1..w7 = a2..a29, w8 = [a30 a31 dB dB], w9..w16 = b0..b31
template <> struct Pair<kFmtQ8, kLayoutGguf> {
    static constexpr int kWords = 17;
    uint32_t x[17];  // x[0..8]: block A codes at w's alignment (zeros facing dA, dB); x[9..16]: block B
    float dxa, dxb;

    __device__ __forceinline__ void set(const uint32_t (&v)[17], int /*p*/ = 0) {
        x[0] = v[0] & 0xffff0000u;
#pragma unroll
        for (int k = 1; k < 8; ++k) x[k] = v[k];
        x[8] = v[8] & 0x0000ffffu;
#pragma unroll
        for (int k = 9; k < 17; ++k) x[k] = v[k];
        dxa = half_lo(v[0]);
        dxb = half_hi(v[8]);
    }
    __device__ __forceinline__ void sums(const uint32_t *w, int &sa, int &sb) const {
        sa = 0;
        sb = 0;
#pragma unroll
        for (int k = 0; k < 9; ++k) sa = dp4a_ss(w[k], x[k], sa);
#pragma unroll
        for (int k = 9; k < 17; ++k) sb = dp4a_ss(w[k], x[k], sb);
    }
    // r: the pair's 17 weight words
    __device__ __forceinline__ float fma_w(const uint32_t (&r)[17], float acc) const {
        int sa, sb;
        sums(r, sa, sb);
        acc = __fmaf_rn(static_cast<float>(sa), __fmul_rn(half_lo(r[0]), dxa), acc);
        acc = __fmaf_rn(static_cast<float>(sb), __fmul_rn(half_hi(r[8]), dxb), acc);
        return acc;
    }
};

// Q4_0, GGUF layout. Weight pair words w[0..8] (36 bytes):
//   w0 = [dA dA qa0 qa1], w1..w3 = qa2..qa13, w4 = [qa14 qa15 dB dB], w5..w8 = qb0..qb15
// low nibble of qa_j is element j, high nibble element j+16.
template <> struct Pair<kFmtQ4, kLayoutGguf> {
    static constexpr int kWords = 9;
    uint32_t xlo[9];  // [0..4]: codes facing the low nibbles of w0..w4 (block A), [5..8]: w5..w8 (block B)
    uint32_t xhi[9];  // the same for the high nibbles
    int inita, initb; // -8 * sum of the block's codes
    float dxa, dxb;

    __device__ __forceinline__ void set(const uint32_t (&v)[17], int /*p*/ = 0) {
        // activation pair bytes: v0 = [dxA dxA x0 x1], v_k = x(4k-2)..x(4k+1), v8 = [x30 x31 dxB dxB]
        xlo[0] = v[0] & 0xffff0000u;         // [0 0 x0 x1]
        xlo[1] = v[1];                       // x2..x5
        xlo[2] = v[2];
        xlo[3] = v[3];
        xlo[4] = v[4] & 0x0000ffffu;         // [x14 x15 0 0]
        xhi[0] = v[4] & 0xffff0000u;         // [0 0 x16 x17]
        xhi[1] = v[5];
        xhi[2] = v[6];
        xhi[3] = v[7];
        xhi[4] = v[8] & 0x0000ffffu;         // [x30 x31 0 0]
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            xlo[5 + k] = v[9 + k];           // block B codes 0..15
            xhi[5 + k] = v[13 + k];          // block B codes 16..31
        }
        uint32_t xa[8], xb[8];
        x_aligned_words(v, xa, xb);
        inita = q4_offset_term(xa);
        initb = q4_offset_term(xb);
        dxa = half_lo(v[0]);
        dxb = half_hi(v[8]);
    }
    __device__ __forceinline__ void sums(const uint32_t *w, int &sa, int &sb) const {
        int la = inita, ha = 0, lb = initb, hb = 0;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            la = dp4a_ss(w[k] & kLoNib, xlo[k], la);
            ha = dp4a_us(w[k] & kHiNib, xhi[k], ha);
        }
#pragma unroll
        for (int k = 5; k < 9; ++k) {
            lb = dp4a_ss(w[k] & kLoNib, xlo[k], lb);
            hb = dp4a_us(w[k] & kHiNib, xhi[k], hb);
        }
        // high nibbles were multiplied in place (16*q): exact division by 16
        sa = la + (ha >> 4);
        sb = lb + (hb >> 4);
    }
    // r: the pair's 9 weight words
    __device__ __forceinline__ float fma_w(const uint32_t (&r)[9], float acc) const {
        int sa, sb;
        sums(r, sa, sb);
        acc = __fmaf_rn(static_cast<float>(sa), __fmul_rn(half_lo(r[0]), dxa), acc);
        acc = __fmaf_rn(static_cast<float>(sb), __fmul_rn(half_hi(r[4]), dxb), acc);
        return acc;
    }
};

// Q8_0, repacked layout: 16 aligned quant words per pair, four 16-byte chunks
// (block A: chunks 0, 1; block B: chunks 2, 3), plus one scale word. Pairs are
// 64 bytes apart, so if every lane loaded its chunks in order, the 8 lanes of a
// 128-bit load phase would hit 2 of the 8 bank quads. The lane owning pair p
// loads chunk s ^ rot at step s, rot = (p >> 1) & 3 (the four lane pairs of a
// phase take four different chunks: 8 distinct bank quads), and holds its
// activation words in the same order. Steps 0, 1 then hold one whole block
// (A when rot < 2) and steps 2, 3 the other: the block sums are the same integers.
template <> struct Pair<kFmtQ8, kLayoutRepacked> {
    static constexpr int kWords = 16;
    static constexpr int kChunks = 4;
    uint32_t x[16];  // x[4s..4s+3]: the activation words facing chunk s ^ rot
    int rot;
    float dxa, dxb;

    __device__ __forceinline__ static int rotation(int p) { return (p >> 1) & 3; }

    __device__ __forceinline__ void set(const uint32_t (&v)[17], int p = 0) {
        uint32_t xa[8], xb[8];
        x_aligned_words(v, xa, xb);
        uint32_t c[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            c[k] = xa[k];
            c[8 + k] = xb[k];
        }
        rot = rotation(p);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t r0 = c[4 * s + i], r1 = c[4 * (s ^ 1) + i];
                const uint32_t r2 = c[4 * (s ^ 2) + i], r3 = c[4 * (s ^ 3) + i];
                x[4 * s + i] = rot == 0 ? r0 : (rot == 1 ? r1 : (rot == 2 ? r2 : r3));
            }
        }
        dxa = half_lo(v[0]);
        dxb = half_hi(v[8]);
    }
    // wq: the weight words in load order (chunk s ^ rot at words 4s..4s+3)
    __device__ __forceinline__ void sums(const uint32_t *wq, int &sa, int &sb) const {
        int lo = 0, hi = 0;  // steps 0, 1 and steps 2, 3
#pragma unroll
        for (int k = 0; k < 8; ++k) lo = dp4a_ss(wq[k], x[k], lo);
#pragma unroll
        for (int k = 8; k < 16; ++k) hi = dp4a_ss(wq[k], x[k], hi);
        sa = rot < 2 ? lo : hi;
        sb = rot < 2 ? hi : lo;
    }
    // wq: shared-memory address of the pair's 16 quant words (16-byte aligned); ws: its scale word
    __device__ __forceinline__ float fma_pair(uint32_t wq, uint32_t ws, float acc) const {
        uint32_t r[16];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint4 t = lds128(wq + 16u * static_cast<uint32_t>(s ^ rot));
            r[4 * s] = t.x;
            r[4 * s + 1] = t.y;
            r[4 * s + 2] = t.z;
            r[4 * s + 3] = t.w;
        }
        int sa, sb;
        sums(r, sa, sb);
        acc = __fmaf_rn(static_cast<float>(sa), __fmul_rn(half_lo(ws), dxa), acc);
        acc = __fmaf_rn(static_cast<float>(sb), __fmul_rn(half_hi(ws), dxb), acc);
        return acc;
    }
};

// Q4_0, repacked layout: 8 aligned quant words per pair, two 16-byte chunks
// (block A, block B) 32 bytes apart from pair to pair, plus one scale word. The
// lane owning pair p loads its chunks in swapped order when rot = (p >> 2) & 1
// is 1 (8 distinct bank quads per 128-bit load phase) and holds its activation
// words and offset terms in the same order; the block sums are the same integers.
template <> struct Pair<kFmtQ4, kLayoutRepacked> {
    static constexpr int kWords = 8;
    static constexpr int kChunks = 2;
    uint32_t xlo[8], xhi[8];  // words 4s..4s+3: facing chunk s ^ rot
    int init0, init1;         // the -8 offset terms of chunk 0 ^ rot and 1 ^ rot
    int rot;
    float dxa, dxb;

    __device__ __forceinline__ static int rotation(int p) { return (p >> 2) & 1; }

    __device__ __forceinline__ void set(const uint32_t (&v)[17], int p = 0) {
        uint32_t xa[8], xb[8];
        x_aligned_words(v, xa, xb);
        rot = rotation(p);
        const bool sw = rot != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            xlo[k] = sw ? xb[k] : xa[k];
            xhi[k] = sw ? xb[4 + k] : xa[4 + k];
            xlo[4 + k] = sw ? xa[k] : xb[k];
            xhi[4 + k] = sw ? xa[4 + k] : xb[4 + k];
        }
        const int ia = q4_offset_term(xa), ib = q4_offset_term(xb);
        init0 = sw ? ib : ia;
        init1 = sw ? ia : ib;
        dxa = half_lo(v[0]);
        dxb = half_hi(v[8]);
    }
    // wq: the weight words in load order (chunk s ^ rot at words 4s..4s+3)
    __device__ __forceinline__ void sums(const uint32_t *wq, int &sa, int &sb) const {
        int l0 = init0, h0 = 0, l1 = init1, h1 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            l0 = dp4a_ss(wq[k] & kLoNib, xlo[k], l0);
            h0 = dp4a_us(wq[k] & kHiNib, xhi[k], h0);
            l1 = dp4a_ss(wq[4 + k] & kLoNib, xlo[4 + k], l1);
            h1 = dp4a_us(wq[4 + k] & kHiNib, xhi[4 + k], h1);
        }
        const int s0 = l0 + (h0 >> 4), s1 = l1 + (h1 >> 4);
        sa = rot ? s1 : s0;
        sb = rot ? s0 : s1;
    }
    __device__ __forceinline__ float fma_pair(uint32_t wq, uint32_t ws, float acc) const {
        uint32_t r[8];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint4 t = lds128(wq + 16u * static_cast<uint32_t>(s ^ rot));
            r[4 * s] = t.x;
            r[4 * s + 1] = t.y;
            r[4 * s + 2] = t.z;
            r[4 * s + 3] = t.w;
        }
        int sa, sb;
        sums(r, sa, sb);
        acc = __fmaf_rn(static_cast<float>(sa), __fmul_rn(half_lo(ws), dxa), acc);
        acc = __fmaf_rn(static_cast<float>(sb), __fmul_rn(half_hi(ws), dxb), acc);
        return acc;
    }
};

// ------------------------------------------------- single-block (plain path)
// Blocks at any 2-byte aligned address: 16-bit loads, aligned words assembled
// in registers. Used by the plain kernel (shapes the pipelined kernel does not
// take) and by its debug counterpart.
__device__ __forceinline__ uint32_t ld_u16_pair(const uint16_t *p) {
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 16);
}

// activation block at xb (34 bytes, 2-byte aligned): aligned code words + scale
__device__ __forceinline__ void load_x_block(const uint8_t *xb, uint32_t (&xw)[8], float &dx) {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(xb);
    dx = __half2float(__ushort_as_half(h[0]));
#pragma unroll
    for (int k = 0; k < 8; ++k) xw[k] = ld_u16_pair(h + 1 + 2 * k);
}

template <int FMT> struct Block;

template <> struct Block<kFmtQ8> {
    // quant words from a GGUF block (2-byte aligned) or an aligned repacked slot
    __device__ __forceinline__ static void load_gguf(const uint8_t *blk, uint32_t (&q)[8], float &d) {
        const uint16_t *h = reinterpret_cast<const uint16_t *>(blk);
        d = __half2float(__ushort_as_half(h[0]));
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = ld_u16_pair(h + 1 + 2 * k);
    }
    __device__ __forceinline__ static void load_repacked(const uint8_t *qs, const uint8_t *sc, uint32_t (&q)[8],
                                                         float &d) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(qs);
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = w[k];
        d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(sc)));
    }
    __device__ __forceinline__ static int dot(const uint32_t (&q)[8], const uint32_t (&xw)[8]) {
        int s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = dp4a_ss(q[k], xw[k], s);
        return s;
    }
};

template <> struct Block<kFmtQ4> {
    __device__ __forceinline__ static void load_gguf(const uint8_t *blk, uint32_t (&q)[8], float &d) {
        const uint16_t *h = reinterpret_cast<const uint16_t *>(blk);
        d = __half2float(__ushort_as_half(h[0]));
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = ld_u16_pair(h + 1 + 2 * k);
#pragma unroll
        for (int k = 4; k < 8; ++k) q[k] = 0;
    }
    __device__ __forceinline__ static void load_repacked(const uint8_t *qs, const uint8_t *sc, uint32_t (&q)[8],
                                                         float &d) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(qs);
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = w[k];
#pragma unroll
        for (int k = 4; k < 8; ++k) q[k] = 0;
        d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(sc)));
    }
    // q[0..3]: the 16 qs bytes; element j = low nibble of qs_j, element j+16 = high nibble
    __device__ __forceinline__ static int dot(const uint32_t (&q)[8], const uint32_t (&xw)[8]) {
        int lo = q4_offset_term(xw), hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            lo = dp4a_ss(q[k] & kLoNib, xw[k], lo);
            hi = dp4a_ss((q[k] >> 4) & kLoNib, xw[4 + k], hi);
        }
        return lo + hi;
    }
};

}  // namespace zdmmv
