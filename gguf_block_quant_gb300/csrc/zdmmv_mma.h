// zdmmv_mma.h -- host-side declarations of the tensor-core batched DMMV (not
// part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace zdmmv {

// Batched DMMV on the integer tensor cores (GGUF layout, 2..8 vectors):
// arguments, plan (false when the kernel does not take the shape) and launchers.
struct MmaArgs {
    const uint8_t *w;    // GGUF rows
    const uint8_t *xq;   // [batch][nb] Q8_0 activation blocks
    float *y;            // [batch][y_stride] outputs
    uint32_t *fault;     // device fault word
    int64_t rows;
    int64_t y_stride;    // floats between vectors' outputs
    int32_t nb;          // blocks per row
    int32_t batch;
    int32_t cb;          // blocks per row in one stage
    int32_t nchunks;     // stages per 16-row slab
    int32_t pitch;       // shared-memory bytes per staged row
    int32_t x_region;    // bytes holding the staged activation, later the partial sums
};
struct MmaPlan {
    int warps;           // consumer warps (8 or 16)
    int stages;
    int cb, nchunks, pitch, x_region;
    int smem_bytes;
};
bool mma_plan(int fmt, int layout, int64_t rows, int64_t cols, int batch, MmaPlan *out);

// Shared by the tensor-core kernels. The weight rows (row_bytes each) as a 2D
// tensor map of 8-byte elements with a box of {pitch / 8, box_rows}, cached per
// calling thread. And the chunking of a row of nb blocks of bb bytes into the
// fewest tensor copies whose shared-memory pitch (at most max_pitch bytes) is 4
// mod 8 words (false when none fits).
cudaError_t weight_map(const uint8_t *w, int64_t rows, int64_t row_bytes, int pitch, int box_rows,
                       CUtensorMap *out);
bool weight_chunk_plan(int nb, int bb, int max_pitch, int *cb, int *nchunks, int *pitch);
cudaError_t launch_mma_q8(const MmaArgs &a, const MmaPlan &p, cudaStream_t st, bool pdl);
cudaError_t launch_mma_q4(const MmaArgs &a, const MmaPlan &p, cudaStream_t st, bool pdl);

}  // namespace zdmmv
