// gemv_q6k.cu -- instantiates the matvec kernels for one weight format
// (one translation unit per format so the builds run in parallel).
#include "gemv_impl.cuh"

namespace qmm {

GemvKernel gemv_pick_q6k(bool q8, int NB, int R) {
    return q8 ? gemv_pick<FMT_Q6_K, true>(NB, R) : gemv_pick<FMT_Q6_K, false>(NB, R);
}

}  // namespace qmm
