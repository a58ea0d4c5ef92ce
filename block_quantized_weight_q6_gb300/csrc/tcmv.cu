// tcmv.cu -- host side of the tensor-core matvec (occupancy, launch) and the
// two small kernels that lay the activations out as its B operand.
#include <cuda_bf16.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "quant.cuh"

namespace qmm {

namespace {

TcmvKernel pick(int fmt, bool q8, int NB, int S) {
    if (fmt == FMT_Q6_K) return tcmv_pick_q6k(q8, NB, S);
    if (fmt == FMT_Q4_0) return tcmv_pick_q4_0(q8, NB, S);
    if (fmt == FMT_Q8_0) return tcmv_pick_q8_0(q8, NB, S);
    return nullptr;
}

uint32_t smem_of(int fmt, int NB, int S) {
    if (fmt == FMT_Q6_K) return tcmv_smem_q6k(NB, S);
    if (fmt == FMT_Q4_0) return tcmv_smem_q4_0(NB, S);
    if (fmt == FMT_Q8_0) return tcmv_smem_q8_0(NB, S);
    return 0;
}

// element offset of activation column c, K index k in the tile: per 256-wide
// stage, core matrices [c / 8][(k % 256) / 8][c % 8][k % 8]
__device__ __forceinline__ int64_t tile_off(int ncol, int c, int64_t k) {
    return (k >> 8) * (static_cast<int64_t>(ncol) * 256) + (c >> 3) * 2048 + ((k & 255) >> 3) * 64 +
           (c & 7) * 8;
}

__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_val(uint32_t h) { return __uint_as_float(h << 16); }

// one thread per 8 consecutive tile elements (16 bytes): tile column c,
// K indices k0..k0+7
__global__ void x_tile_kernel(const void* __restrict__ x, int x_bf16, int B, int64_t K, int S,
                              int ncol, int64_t nst, uint16_t* __restrict__ xt, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_X_TILE);
    const int64_t units = nst * ncol * 32;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // u enumerates [stage][c / 8][k8][c % 8]: consecutive threads write
        // consecutive 16-byte pieces
        const int c8 = static_cast<int>(u & 7);
        const int64_t k8 = (u >> 3) & 31;
        const int64_t rest = u >> 8;
        const int cg = static_cast<int>(rest % (ncol / 8));
        const int64_t stg = rest / (ncol / 8);
        const int c = cg * 8 + c8;
        const int64_t k0 = stg * 256 + k8 * 8;
        const int b = c / S, j = c % S;
        uint32_t h[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float f = 0.0f;
            const int64_t k = k0 + t;
            if (b < B && k < K) {
                if (x_bf16)
                    f = bf16_val(static_cast<const uint16_t*>(x)[b * K + k]);
                else
                    f = static_cast<const float*>(x)[b * K + k];
            }
            if (S == 1) {
                h[t] = bf16_bits(f);
            } else {
                // f = hi + mid + lo exactly (8 + 8 + 8 significant bits)
                const uint32_t hi = bf16_bits(f);
                const float r1 = f - bf16_val(hi);
                const uint32_t mid = bf16_bits(r1);
                const uint32_t lo = bf16_bits(r1 - bf16_val(mid));
                h[t] = j == 0 ? hi : (j == 1 ? mid : lo);
            }
        }
        uint4* o = reinterpret_cast<uint4*>(xt + tile_off(ncol, c, k0));
        *o = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                        h[6] | (h[7] << 16));
    }
}

// one thread per (tile column r, 32-wide block kb): quantizes row r < B of
// the activations and writes its codes (exact bf16) and scale; columns
// B..ncol-1 and blocks past K are zeros
__global__ void q8_tile_kernel(const void* __restrict__ x, int x_bf16, int B, int64_t K, int NB,
                               int ncol, int64_t nst, uint16_t* __restrict__ xt,
                               float* __restrict__ xs, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_QUANTIZE);
    const int64_t nkb = nst * 8;
    const int64_t units = nkb * ncol;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(u % ncol);
        const int64_t kb = u / ncol;
        int q[32];
        float s = 0.0f;
        if (r < B && kb < K / 32) {
            float v[32];
            load_x32(x, x_bf16, K, r, kb, v);
            s = quantize_block32(v, q);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = 0;
        }
        if (r < NB) xs[kb * NB + r] = s;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
            uint32_t h[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) h[t] = bf16_bits(static_cast<float>(q[8 * k8 + t]));
            uint4* o = reinterpret_cast<uint4*>(xt + tile_off(ncol, r, kb * 32 + 8 * k8));
            *o = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                            h[6] | (h[7] << 16));
        }
    }
}

int grid_for(int64_t units, int threads) {
    int64_t blocks = (units + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

int tcmv_occupancy(int fmt, bool q8, int NB, int S) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, fmt, q8 ? 1 : 0, NB, S, 0);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int occ = 0;
    TcmvKernel k = pick(fmt, q8, NB, S);
    const uint32_t smem = smem_of(fmt, NB, S);
    if (k && smem) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) == cudaSuccess &&
            cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kTcThreads, smem) != cudaSuccess)
            occ = 0;
    }
    (void)cudaGetLastError();
    cache[key] = occ;
    return occ;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

int row_slot_bytes(int fmt) { return fmt == FMT_Q6_K ? 240 : (fmt == FMT_Q4_0 ? 176 : 304); }

}  // namespace

cudaError_t tcmv_launch(int fmt, bool q8, int NB, int S, int grid, cudaStream_t s,
                        const TcmvArgs& a) {
    TcmvKernel k = pick(fmt, q8, NB, S);
    if (!k || tcmv_occupancy(fmt, q8, NB, S) <= 0) return cudaErrorInvalidValue;
    // W as [N / 8][8 * rowbytes] bytes of 16-bit elements: the pitch of 8 rows
    // is a multiple of 16 bytes for every even row size; a box is one row
    // slot wide and 16 groups of 8 rows high
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    if (a.n8 > 0) {
        EncodeTiledFn enc = encode_fn();
        if (!enc) return cudaErrorNotSupported;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(4 * a.rowbytes),
                                    static_cast<cuuint64_t>(a.n8 / 8)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(8 * a.rowbytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_slot_bytes(fmt) / 2), 16u};
        const cuuint32_t es[2] = {1u, 1u};
        if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(a.W), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = launch_pdl(k, dim3(grid), dim3(kTcThreads), smem_of(fmt, NB, S), s, a, map);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t x_tile_launch(const void* x, int x_bf16, int B, int64_t K, int S, int ncol,
                          int64_t nst, uint16_t* xt, cudaStream_t s, DevState st) {
    const int threads = 256;
    cudaError_t e = launch_pdl(x_tile_kernel, dim3(grid_for(nst * ncol * 32, threads)),
                               dim3(threads), 0, s, x, x_bf16, B, K, S, ncol, nst, xt, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t q8_tile_launch(const void* x, int x_bf16, int B, int64_t K, int NB, int ncol,
                           int64_t nst, uint16_t* xt, float* xs, cudaStream_t s, DevState st) {
    const int threads = 128;
    cudaError_t e = launch_pdl(q8_tile_kernel, dim3(grid_for(nst * 8 * ncol, threads)),
                               dim3(threads), 0, s, x, x_bf16, B, K, NB, ncol, nst, xt, xs, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmm
