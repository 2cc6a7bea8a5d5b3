// zdmmv_acc_q4.cu -- the pipelined Q4_0 DMMV with the accumulate epilogue (instantiations).
#include "zdmmv_tma.cuh"

namespace zdmmv {

cudaError_t launch_acc_q4(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl) {
    return launch_epi_fmt<kFmtQ4, 2>(a, p, layout, ctas, st, pdl);
}

}  // namespace zdmmv
