// zdmmv_argmax_q8.cu -- the pipelined Q8_0 DMMV with the argmax epilogue (instantiations).
#include "zdmmv_tma.cuh"

namespace zdmmv {

cudaError_t launch_argmax_q8(const DmmvArgs &a, const TmaPlan &p, int layout, int ctas, cudaStream_t st, bool pdl) {
    return launch_argmax_fmt<kFmtQ8>(a, p, layout, ctas, st, pdl);
}

}  // namespace zdmmv
