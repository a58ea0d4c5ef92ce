// tcmv_q4_0.cu -- instantiates the tensor-core matvec for one weight format
// (one translation unit per format so the builds run in parallel).
#include "tcmv.cuh"

namespace qmm {

TcmvKernel tcmv_pick_q4_0(bool q8, int NB, int S) { return tcmv_pick<FMT_Q4_0>(q8, NB, S); }
uint32_t tcmv_smem_q4_0(int NB, int S) { return tcmv_smem_of<FMT_Q4_0>(NB, S); }

}  // namespace qmm
