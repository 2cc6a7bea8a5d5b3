// zdmmv_swiglu_q8.cu -- the pipelined Q8_0 DMMV with the SwiGLU pair epilogue (instantiations).
#include "zdmmv_tma.cuh"

namespace zdmmv {

cudaError_t launch_swiglu_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                             cudaStream_t st, bool pdl) {
    return launch_epi_fmt<kFmtQ8, 3>(a, p, layout, ctas_per_slot, st, pdl, slots);
}

int swiglu_ctas_per_sm_q8(int layout, const TmaPlan &p) { return tma_ctas_per_sm_fmt<kFmtQ8, 3>(layout, p); }

}  // namespace zdmmv
