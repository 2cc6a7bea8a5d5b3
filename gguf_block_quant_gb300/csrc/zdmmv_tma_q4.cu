// zdmmv_tma_q4.cu -- instantiations of the TMA-pipelined DMMV kernel for Q4_0 weights.
#include "zdmmv_batch.cuh"
#include "zdmmv_tma.cuh"

namespace zdmmv {

cudaError_t launch_tma_q4(const DmmvArgs &a, const TmaPlan &p, int layout, bool fused_x, int ctas_per_slot,
                          int slots, cudaStream_t st, bool pdl) {
    return launch_tma_fmt<kFmtQ4>(a, p, layout, fused_x, ctas_per_slot, slots, st, pdl);
}

int tma_ctas_per_sm_q4(int layout, const TmaPlan &p) { return tma_ctas_per_sm_fmt<kFmtQ4>(layout, p); }

cudaError_t launch_batch_q4(const DmmvArgs &a, const BatchPlan &p, int layout, int ctas, cudaStream_t st,
                            bool pdl) {
    return launch_batch_fmt<kFmtQ4>(a, layout, p.g, p.bpt, p.vb, p.stages, p.smem_bytes, ctas, st, pdl);
}

}  // namespace zdmmv
