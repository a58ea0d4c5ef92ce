// gemv_q8_0.cu -- instantiates the matvec kernels for one weight format
// (one translation unit per format so the builds run in parallel).
#include "gemv_impl.cuh"

namespace qmm {

GemvKernel gemv_pick_q8_0(bool q8, int NB, int R) {
    return q8 ? gemv_pick<FMT_Q8_0, true>(NB, R) : gemv_pick<FMT_Q8_0, false>(NB, R);
}

}  // namespace qmm
