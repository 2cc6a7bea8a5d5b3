// zdmmv_mma.h -- host-side declarations of the tensor-core kernels (not part of
// the public C ABI): the weight tensor map they share, and each kernel's plan and
// launcher.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace zdmmv {

// The weight rows (row_bytes each) as a 2D tensor map of 8-byte elements with a
// box of {pitch / 8, box_rows}, cached per calling thread.
cudaError_t weight_map(const uint8_t *w, int64_t rows, int64_t row_bytes, int pitch, int box_rows,
                       CUtensorMap *out);

// The DMMV with an fp32 activation taken as is (no quantization) on the fp16
// tensor cores (GGUF rows of 256-column multiples, tall matrices): plan (false
// when it does not take the shape) and launcher (Xf32MmaArgs: zdmmv_xf32_mma.cuh).
struct Xf32MmaArgs;
struct Xf32MmaPlan {
    int cb, nchunks, pitch;  // blocks per stage row, stages per row group, staged row pitch (bytes)
    int stages, smem_bytes;
};
bool xf32_mma_plan(int fmt, int layout, int64_t rows, int64_t cols, Xf32MmaPlan *out);
cudaError_t launch_xf32_mma(int fmt, const Xf32MmaArgs &a, const Xf32MmaPlan &p, int slots, cudaStream_t st,
                            bool pdl);

// The batched DMMV (1..8 Q8_0 vectors, GGUF rows of 256-column multiples) on
// the fp16 tensor cores: plan (false when it does not take the shape) and
// launcher (BmmaArgs: zdmmv_bmma.cuh).
struct BmmaArgs;
struct BmmaPlan {
    int nchunks, pitch;   // stages per 32-row group, staged row pitch (bytes)
    int red_bufs;         // buffers of warp partial sums (1 or 2)
    int stages, smem_bytes;
};
bool bmma_plan(int fmt, int layout, int64_t rows, int64_t cols, int batch, BmmaPlan *out);
cudaError_t launch_bmma(int fmt, const BmmaArgs &a, const BmmaPlan &p, bool fused_x, cudaStream_t st, bool pdl);

}  // namespace zdmmv
