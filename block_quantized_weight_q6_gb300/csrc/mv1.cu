// mv1.cu -- instantiations and launch of the batch-1 CUDA-core matvec
// (mv1.cuh).
#include "mv1.cuh"

namespace qmm {

bool mv1_supported(int fmt, int64_t K) {
    if (K <= 0) return false;
    if (fmt == FMT_Q6_K) return K % 256 == 0;  // (the dispatch also wants 16-byte rows)
    return (fmt == FMT_Q4_0 || fmt == FMT_Q8_0) && K % 256 == 0;
}

template <int FMT>
static cudaError_t mv1_prepare(int* occ) {
    static int done = 0, o = 0;
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(mv1_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             mv1_smem_bytes<FMT>());
        if (e != cudaSuccess) return e;
        // the same shared/L1 split as the tensor-core kernels, so that
        // consecutive launches need not change it
        e = cudaFuncSetAttribute(mv1_kernel<FMT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, mv1_kernel<FMT>, kMv1Warps * 32,
                                                          mv1_smem_bytes<FMT>());
        if (e != cudaSuccess) return e;
        done = 1;
    }
    if (occ) *occ = o;
    return cudaSuccess;
}

int mv1_occupancy(int fmt) {
    int o = 0;
    cudaError_t e = fmt == FMT_Q6_K ? mv1_prepare<FMT_Q6_K>(&o)
                  : fmt == FMT_Q4_0 ? mv1_prepare<FMT_Q4_0>(&o)
                                    : mv1_prepare<FMT_Q8_0>(&o);
    return e == cudaSuccess ? o : 0;
}

cudaError_t mv1_launch(int fmt, int grid, cudaStream_t s, const Mv1Group& g) {
    const dim3 block(kMv1Warps * 32);
    switch (fmt) {
        case FMT_Q6_K:
            return launch_pdl(mv1_kernel<FMT_Q6_K>, dim3(grid), block, mv1_smem_bytes<FMT_Q6_K>(), s, g);
        case FMT_Q4_0:
            return launch_pdl(mv1_kernel<FMT_Q4_0>, dim3(grid), block, mv1_smem_bytes<FMT_Q4_0>(), s, g);
        case FMT_Q8_0:
            return launch_pdl(mv1_kernel<FMT_Q8_0>, dim3(grid), block, mv1_smem_bytes<FMT_Q8_0>(), s, g);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
