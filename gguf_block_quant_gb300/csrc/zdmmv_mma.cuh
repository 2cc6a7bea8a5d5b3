// zdmmv_mma.cuh -- pieces shared by the tensor-core DMMV kernels (the batched
// kernel, zdmmv_bmma.cuh, and the fp32-activation kernel, zdmmv_xf32_mma.cuh),
// for sm_103a.
//
// Both stream the weights with one 2D tensor copy per stage: the GGUF rows as a
// 2D tensor of 8-byte elements, a box of a group of 16-row slabs by a chunk of
// blocks, whose shared-memory pitch is 4 mod 8 words so that the 8 rows of a
// fragment load (one per lane quad) fall in 8 distinct bank quads; rows and
// columns past the matrix are zero-filled by the copy. (Sixteen row-by-row bulk
// copies per stage were measured first: about 50 ns of copy-engine time each kept
// HBM below half its rate.)
//
// Lane (g, t) of a warp (g = lane / 4, t = lane % 4) takes the aligned words of a
// GGUF block pair (68 or 36 bytes, 4-byte aligned): in it the odd block's codes
// are aligned words and the even block's codes start 2 bytes in, so for the even
// block the last lane of a quad combines the two stray halves (the first two
// codes, in the word holding the scale, and the last two) with one byte permute.
#pragma once

#include <cuda.h>

#include "zdmmv.h"
#include "zdmmv_mma.h"
#include "zdmmv_tma.cuh"

namespace zdmmv {

constexpr int kMmaRows = 16;  // rows per slab (the MMA's M)

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

// Byte permute that finishes lane t's second word of an even block: identity,
// except on the last lane of a quad, which keeps bytes 0, 1 of its word (the
// block's last two codes) and takes bytes 2, 3 of the pair's first word (the
// block's first two codes).
__device__ __forceinline__ uint32_t mma_even_sel(int t) { return t == 3 ? 0x7610u : 0x3210u; }

template <int NW>
__device__ __forceinline__ void mma_consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

}  // namespace zdmmv
