// zdmmv_mma.h -- host-side declarations shared by the tensor-core kernels (not
// part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace zdmmv {

// The weight rows (row_bytes each) as a 2D tensor map of 8-byte elements with a
// box of {pitch / 8, box_rows}, cached per calling thread.
cudaError_t weight_map(const uint8_t *w, int64_t rows, int64_t row_bytes, int pitch, int box_rows,
                       CUtensorMap *out);

}  // namespace zdmmv
