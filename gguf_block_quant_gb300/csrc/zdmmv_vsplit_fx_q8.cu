// zdmmv_vsplit_fx_q8.cu -- the Q8_0 batched DMMV with vectors split over warps and
// the activations quantized in the prologue (instantiations).
#include "zdmmv_vsplit.cuh"

namespace zdmmv {

cudaError_t launch_vsplit_fx_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int v, int nvg, int max_per_sm,
                                cudaStream_t st, bool pdl) {
    return launch_vsplit_fmt<kFmtQ8, true>(a, p, layout, v, nvg, max_per_sm, st, pdl);
}

}  // namespace zdmmv
