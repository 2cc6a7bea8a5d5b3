// zdmmv_mma.cu -- the weight tensor map shared by the tensor-core kernels.
#include <cudaTypedefs.h>

#include "zdmmv.h"
#include "zdmmv_mma.cuh"

namespace zdmmv {

namespace {
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); nullptr when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}
}  // namespace

// The weight rows as a 2D tensor of 8-byte elements ({row_bytes / 8, rows},
// row stride row_bytes), box {pitch / 8, box_rows}; the last few maps of the
// calling thread are kept, so repeated calls on the same matrix encode nothing.
cudaError_t weight_map(const uint8_t *w, int64_t rows, int64_t row_bytes, int pitch, int box_rows,
                       CUtensorMap *out) {
    struct Entry {
        const uint8_t *w;
        int64_t rows, row_bytes;
        int pitch, box_rows;
        CUtensorMap map;
    };
    constexpr int kKeep = 8;
    thread_local Entry cache[kKeep];
    thread_local int next = 0;
    for (const Entry &e : cache) {
        if (e.w == w && e.rows == rows && e.row_bytes == row_bytes && e.pitch == pitch && e.box_rows == box_rows) {
            *out = e.map;
            return cudaSuccess;
        }
    }
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 8), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pitch / 8), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem_strides[2] = {1, 1};
    Entry &e = cache[next];
    if (enc(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(w), dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        e.w = nullptr;
        return cudaErrorInvalidValue;
    }
    e.w = w;
    e.rows = rows;
    e.row_bytes = row_bytes;
    e.pitch = pitch;
    e.box_rows = box_rows;
    next = (next + 1) % kKeep;
    *out = e.map;
    return cudaSuccess;
}

}  // namespace zdmmv
