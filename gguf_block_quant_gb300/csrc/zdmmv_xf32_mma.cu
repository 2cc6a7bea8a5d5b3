// zdmmv_xf32_mma.cu -- plan, weight tensor map and instantiations of the
// fp32-activation DMMV on the fp16 tensor cores.
#include "zdmmv_internal.h"
#include "zdmmv_xf32_mma.cuh"

namespace zdmmv {

namespace {
constexpr int kXmWarps = 8;
constexpr int kXmSmemTwoPerSm = 110 * 1024;  // two CTAs per SM
constexpr int kXmSmemMax = 220 * 1024;       // one CTA per SM
constexpr int kXmMaxStages = 8;
constexpr int kXmMinGroupsPerSm = 4;

int fmt_block_bytes(int fmt) { return fmt == kFmtQ8 ? 34 : (fmt == kFmtQ4 ? 18 : 0); }
}  // namespace

// GGUF rows of 256-column multiples (whole 16-byte row strides), at least
// kXmMinGroupsPerSm whole row groups (kXmWarps x 16 rows, the height of a tensor
// copy) per SM. A stage is kXmWarps x 16 rows by a chunk of 8 blocks; two CTAs
// per SM where three stages fit beside the activation fragments (256 bytes per
// block), else one; then as many stages as fit (2, 3, 4, 6 or 8).
bool xf32_mma_plan(int fmt, int layout, int64_t rows, int64_t cols, Xf32MmaPlan *out) {
    if (layout != kLayoutGguf || fmt_block_bytes(fmt) == 0) return false;
    constexpr int kGroupRows = kXmWarps * kMmaRows;
    if (rows < kGroupRows || cols <= 0 || cols % 256 != 0) return false;
    // tall matrices only: with fewer than kXmMinGroupsPerSm row groups per SM the
    // 128-row groups leave SMs idle or unevenly loaded, and the scalar kernel's
    // finer row split is faster (Q8_0 14336 x 4096: 21.9 against 14.4 us)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return false;
    if ((rows + kGroupRows - 1) / kGroupRows < static_cast<int64_t>(kXmMinGroupsPerSm) * sms) return false;
    const int nb = static_cast<int>(cols / kQK);
    const int fixed = kBarrierBytes + nb * kXmFragBytes;
    Xf32MmaPlan p{};
    p.cb = kXmChunkBlocks;
    p.nchunks = nb / kXmChunkBlocks;
    p.pitch = kXmChunkBlocks * fmt_block_bytes(fmt);
    const int stage = kGroupRows * p.pitch;
    // two CTAs per SM where three stages fit beside the fragments, else one CTA per SM
    // (three CTAs per SM with three stages each measured no faster on the LM head)
    const int budget = fixed + 3 * stage <= kXmSmemTwoPerSm ? kXmSmemTwoPerSm : kXmSmemMax;
    int stages = (budget - fixed) / stage;
    stages = stages > kXmMaxStages ? kXmMaxStages : stages;
    stages = stages >= 8 ? 8 : (stages >= 6 ? 6 : (stages >= 4 ? 4 : stages));  // instantiated: 2, 3, 4, 6, 8
    if (stages >= 2) {
        p.stages = stages;
        p.smem_bytes = fixed + stages * stage;
        *out = p;
        return true;
    }
    return false;
}

template <int FMT>
cudaError_t launch_xf32_mma_fmt(const Xf32MmaArgs &a, const Xf32MmaPlan &p, int slots, cudaStream_t st, bool pdl) {
    CUtensorMap map;
    const cudaError_t e = weight_map(a.w, a.rows, static_cast<int64_t>(a.nb) * Fmt<FMT>::kBlockBytes, p.pitch,
                                     kXmWarps * kMmaRows, &map);
    if (e != cudaSuccess) return e;
#define ZDMMV_XM(S_) \
    if (p.stages == S_) return Xf32MmaInst<FMT, kXmWarps, S_>::launch(a, map, p.smem_bytes, slots, st, pdl);
    ZDMMV_XM(2)
    ZDMMV_XM(3)
    ZDMMV_XM(4)
    ZDMMV_XM(6)
    ZDMMV_XM(8)
#undef ZDMMV_XM
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_xf32_mma(int fmt, const Xf32MmaArgs &a, const Xf32MmaPlan &p, int slots, cudaStream_t st,
                            bool pdl) {
    return fmt == kFmtQ8 ? launch_xf32_mma_fmt<kFmtQ8>(a, p, slots, st, pdl)
                         : launch_xf32_mma_fmt<kFmtQ4>(a, p, slots, st, pdl);
}

}  // namespace zdmmv
