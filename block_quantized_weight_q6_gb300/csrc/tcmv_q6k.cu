// tcmv_q6k.cu -- instantiates the tensor-core matvec for one weight format
// (one translation unit per format so the builds run in parallel).
#include "tcmv.cuh"

namespace qmm {

TcmvKernel tcmv_pick_q6k(bool q8, int NB, int S) { return tcmv_pick<FMT_Q6_K>(q8, NB, S); }
uint32_t tcmv_smem_q6k(int NB, int S) { return tcmv_smem_of<FMT_Q6_K>(NB, S); }

}  // namespace qmm
