// zdmmv_bmma.cu -- plan, weight tensor map and instantiations of the batched
// DMMV on the fp16 tensor cores.
#include "zdmmv_internal.h"
#include "zdmmv_bmma.cuh"

namespace zdmmv {

namespace {
constexpr int kBmMaxStages = 8;

int bm_block_bytes(int fmt) { return fmt == kFmtQ8 ? 34 : (fmt == kFmtQ4 ? 18 : 0); }
}  // namespace

// GGUF rows of 256-column multiples (whole 16-byte row strides), at least 32
// rows and 1280 to 4096 columns (a box inside the matrix; the fragment build's
// registers). A stage is 32
// rows by a chunk of 32 blocks, its shared-memory pitch the chunk plus 16 bytes
// (4 mod 8 words; the extra bytes are the next chunk's, or zero-filled past the
// row). Beside the stages: the activation fragments and table of every block of
// the padded row, and two buffers of warp partial sums (one where two would cost
// a stage below three). Then as many stages as fit (2, 3, 4, 6 or 8).
bool bmma_plan(int fmt, int layout, int64_t rows, int64_t cols, int batch, BmmaPlan *out) {
    const int bb = bm_block_bytes(fmt);
    if (layout != kLayoutGguf || bb == 0) return false;
    if (rows < 1 || cols <= 0 || cols % 256 != 0 || batch < 1 || batch > 8) return false;
    if (cols / kQK > kBmMaxBlocks) return false;  // the fragment build holds a row's blocks in registers
    // every tensor copy's box (32 rows by the staged pitch) inside the matrix
    if (rows < kBmGroupRows || (cols / kQK) * bb < kBmChunkBlocks * bb + 16) return false;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return false;
    const int nb = static_cast<int>(cols / kQK);
    BmmaPlan p{};
    p.nchunks = (nb + kBmChunkBlocks - 1) / kBmChunkBlocks;
    const int chunk = kBmChunkBlocks * bb;  // 0 mod 8 words for both formats
    p.pitch = chunk + 16;
    const int nb_pad = p.nchunks * kBmChunkBlocks;
    const int64_t fixed0 = kBarrierBytes + static_cast<int64_t>(nb_pad) * (kBmFragBytes + kBmTableBytes);
    const int stage = kBmGroupRows * p.pitch;
    int64_t stages = 0;
    for (int bufs = 2; bufs >= 1; --bufs) {
        const int64_t fixed = fixed0 + static_cast<int64_t>(bufs) * kBmRedBytes;
        stages = fixed < optin ? (optin - fixed) / stage : 0;
        p.red_bufs = bufs;
        if (stages >= 3) break;
    }
    if (stages < 2) return false;
    stages = stages > kBmMaxStages ? kBmMaxStages : stages;
    stages = stages >= 8 ? 8 : (stages >= 6 ? 6 : (stages >= 4 ? 4 : stages));  // instantiated: 2, 3, 4, 6, 8
    p.stages = static_cast<int>(stages);
    p.smem_bytes = static_cast<int>(fixed0 + static_cast<int64_t>(p.red_bufs) * kBmRedBytes + stages * stage);
    *out = p;
    return true;
}

template <int FMT, bool FX>
cudaError_t launch_bmma_fmt(const BmmaArgs &a, const BmmaPlan &p, cudaStream_t st, bool pdl) {
    CUtensorMap map;
    const cudaError_t e = weight_map(a.w, a.rows, static_cast<int64_t>(a.nb) * Fmt<FMT>::kBlockBytes, p.pitch,
                                     kBmGroupRows, &map);
    if (e != cudaSuccess) return e;
#define ZDMMV_BM(S_) \
    if (p.stages == S_) return BmmaInst<FMT, S_, FX>::launch(a, map, p.smem_bytes, st, pdl);
    ZDMMV_BM(2)
    ZDMMV_BM(3)
    ZDMMV_BM(4)
    ZDMMV_BM(6)
    ZDMMV_BM(8)
#undef ZDMMV_BM
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_bmma(int fmt, const BmmaArgs &a, const BmmaPlan &p, bool fused_x, cudaStream_t st, bool pdl) {
    if (fused_x)
        return fmt == kFmtQ8 ? launch_bmma_fmt<kFmtQ8, true>(a, p, st, pdl) : launch_bmma_fmt<kFmtQ4, true>(a, p, st, pdl);
    return fmt == kFmtQ8 ? launch_bmma_fmt<kFmtQ8, false>(a, p, st, pdl) : launch_bmma_fmt<kFmtQ4, false>(a, p, st, pdl);
}

}  // namespace zdmmv
