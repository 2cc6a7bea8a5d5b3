// zdmmv_xf32_q8.cu -- the Q8_0 DMMV with an fp32 (unquantized) activation (instantiations).
#include "zdmmv_xf32.cuh"

namespace zdmmv {

cudaError_t launch_xf32_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas_per_slot, int slots,
                           cudaStream_t st, bool pdl) {
    return launch_xf32_fmt<kFmtQ8>(a, p, layout, ctas_per_slot, slots, st, pdl);
}

cudaError_t launch_xf32_plain_q8(const DmmvArgs &a, int layout, int sms, int slots, cudaStream_t st, bool pdl) {
    return launch_xf32_plain_fmt<kFmtQ8>(a, layout, sms, slots, st, pdl);
}

}  // namespace zdmmv
