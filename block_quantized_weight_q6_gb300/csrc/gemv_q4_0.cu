// gemv_q4_0.cu -- instantiates the matvec kernels for one weight format
// (one translation unit per format so the builds run in parallel).
#include "gemv_impl.cuh"

namespace qmm {

GemvKernel gemv_pick_q4_0(bool q8, int NB, int R) {
    return q8 ? gemv_pick<FMT_Q4_0, true>(NB, R) : gemv_pick<FMT_Q4_0, false>(NB, R);
}

}  // namespace qmm
