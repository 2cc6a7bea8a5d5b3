// zdmmv_mma.cu -- plan, weight tensor map and instantiations of the tensor-core
// batched DMMV.
#include <cstdlib>
#include <cudaTypedefs.h>

#include "zdmmv.h"
#include "zdmmv_mma.cuh"

namespace zdmmv {

namespace {
int env_int(const char *name, int lo, int hi, int dflt) {
    const char *e = std::getenv(name);
    const int v = e ? std::atoi(e) : dflt;
    return (v >= lo && v <= hi) ? v : dflt;
}
int64_t round_up_to(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

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

namespace {
// Fewest chunks per row whose box fits a tensor copy (at most 256 elements, at
// most max_pitch and 2048 bytes, inside the row) at a width of 4 mod 8 words: a
// chunk of a multiple of 8 blocks, plus 16 bytes (zero-filled past the chunk)
// where its width is 0 mod 8. False when no chunking fits.
bool chunk_plan(int nb, int bb, int max_pitch, int *cb_out, int *nchunks_out, int *pitch_out) {
    const int row_bytes = nb * bb;
    for (int nch = 1; nch <= nb / 8; ++nch) {
        const int cb = static_cast<int>(round_up_to((nb + nch - 1) / nch, 8));
        if (cb * (nch - 1) >= nb) continue;
        const int cbytes = cb * bb;
        const int box = (cbytes / 4) % 8 == 4 ? cbytes : cbytes + 16;
        if (box > 2048 || box > max_pitch || box > row_bytes) continue;
        *cb_out = cb;
        *nchunks_out = nch;
        *pitch_out = box;
        return true;
    }
    return false;
}
}  // namespace

bool weight_chunk_plan(int nb, int bb, int max_pitch, int *cb, int *nchunks, int *pitch) {
    return chunk_plan(nb, bb, max_pitch, cb, nchunks, pitch);
}

// GGUF rows of 256-column multiples (whole 16-byte row strides) up to 4096
// columns and at least one 16-row slab: the staged activation, its fragments and
// table (320 bytes per block) and two or more stages share the 227 KB of one CTA.
bool mma_plan(int fmt, int layout, int64_t rows, int64_t cols, int batch, MmaPlan *out) {
    if (layout != kLayoutGguf || (fmt != kFmtQ8 && fmt != kFmtQ4)) return false;
    if (batch < 2 || batch > 8 || rows < kMmaRows || cols <= 0 || cols % 256 != 0 || cols > 4096) return false;
    const int bb = fmt == kFmtQ8 ? 34 : 18;
    const int nb = static_cast<int>(cols / kQK);
    MmaPlan p{};
    p.warps = env_int("ZDMMV_MMA_WARPS", 8, 16, 8) == 16 ? 16 : 8;
    if (!chunk_plan(nb, bb, 2048, &p.cb, &p.nchunks, &p.pitch)) return false;
    const int64_t xbytes = static_cast<int64_t>(batch) * nb * 34;
    const int64_t red = 2ll * p.warps * 512;
    p.x_region = static_cast<int>(round_up_to(xbytes > red ? xbytes : red, 128));
    const int fixed = kBarrierBytes + p.x_region + nb * (kMmaFragBytes + kMmaTableBytes);
    const int stage = kMmaRows * p.pitch;
    constexpr int kSmemMax = 227 * 1024;
    p.stages = env_int("ZDMMV_MMA_STAGES", 2, 6, 6);
    while (p.stages > 2 && fixed + p.stages * stage > kSmemMax) --p.stages;
    p.smem_bytes = fixed + p.stages * stage;
    if (p.smem_bytes > kSmemMax) return false;
    *out = p;
    return true;
}

template <int FMT>
cudaError_t launch_mma(const MmaArgs &a, const MmaPlan &p, cudaStream_t st, bool pdl) {
    CUtensorMap map;
    const cudaError_t e =
        weight_map(a.w, a.rows, static_cast<int64_t>(a.nb) * Fmt<FMT>::kBlockBytes, p.pitch, kMmaRows, &map);
    if (e != cudaSuccess) return e;
    return launch_mma_fmt<FMT>(a, map, p, st, pdl);
}

cudaError_t launch_mma_q8(const MmaArgs &a, const MmaPlan &p, cudaStream_t st, bool pdl) {
    return launch_mma<kFmtQ8>(a, p, st, pdl);
}
cudaError_t launch_mma_q4(const MmaArgs &a, const MmaPlan &p, cudaStream_t st, bool pdl) {
    return launch_mma<kFmtQ4>(a, p, st, pdl);
}

}  // namespace zdmmv
