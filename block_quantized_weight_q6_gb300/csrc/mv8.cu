// mv8.cu -- instantiations and launch of the batch 2-8 matvec on the
// warp-level MMA (mv8.cuh).
#include "mv8.cuh"

namespace qmm {

bool mv8_supported(int fmt, int64_t K) {
    return K > 0 && K % kMv8StageK == 0 && (fmt == FMT_Q4_0 || fmt == FMT_Q8_0 || fmt == FMT_Q6_K);
}

template <int FMT>
static cudaError_t mv8_prepare(int* occ) {
    static int done = 0, o = 0;
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(mv8_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             mv8_smem_bytes<FMT>());
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(mv8_kernel<FMT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, mv8_kernel<FMT>, kMv8Warps * 32,
                                                          mv8_smem_bytes<FMT>());
        if (e != cudaSuccess) return e;
        done = 1;
    }
    if (occ) *occ = o;
    return cudaSuccess;
}

int mv8_occupancy(int fmt) {
    int o = 0;
    cudaError_t e = fmt == FMT_Q6_K ? mv8_prepare<FMT_Q6_K>(&o)
                  : fmt == FMT_Q4_0 ? mv8_prepare<FMT_Q4_0>(&o)
                                    : mv8_prepare<FMT_Q8_0>(&o);
    return e == cudaSuccess ? o : 0;
}

cudaError_t mv8_launch(int fmt, int grid, cudaStream_t s, const Mv1Group& g) {
    const dim3 block(kMv8Warps * 32);
    switch (fmt) {
        case FMT_Q6_K:
            return launch_pdl(mv8_kernel<FMT_Q6_K>, dim3(grid), block, mv8_smem_bytes<FMT_Q6_K>(), s, g);
        case FMT_Q4_0:
            return launch_pdl(mv8_kernel<FMT_Q4_0>, dim3(grid), block, mv8_smem_bytes<FMT_Q4_0>(), s, g);
        case FMT_Q8_0:
            return launch_pdl(mv8_kernel<FMT_Q8_0>, dim3(grid), block, mv8_smem_bytes<FMT_Q8_0>(), s, g);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
