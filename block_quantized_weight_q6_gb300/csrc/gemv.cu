// gemv.cu -- the small kernels around the matvec and the GEMM: the split-K
// reduction, the per-32 activation quantizer (with the GEMM's A-operand
// tiles) and the W_exp plane build.
#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"
#include "quant.cuh"

namespace qmm {

// ------------------------------------------------------------ split-K reduce

__global__ void splitk_reduce_kernel(const float* __restrict__ part, float* __restrict__ y,
                                     int splits, int64_t count, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v = 0.0f;
        for (int s = 0; s < splits; ++s) v += part[s * count + i];
        y[i] = v;
    }
}

// The same for the split matrices of one grouped matvec, in one launch:
// element i of the set belongs to the matrix m with start[m] <= i < start[m + 1].
__global__ void splitk_reduce_set_kernel(const SplitReduceSet r, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < r.total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int m = 0;
        for (int q = 1; q < r.n; ++q)
            if (i >= r.start[q]) m = q;
        const int64_t j = i - r.start[m], count = r.count[m];
        const float* part = r.part[m];
        float v = 0.0f;
        for (int s = 0; s < r.splits[m]; ++s) v += part[s * count + j];
        r.y[m][j] = v;
    }
}

cudaError_t splitk_reduce_set_launch(const SplitReduceSet& r, cudaStream_t s, DevState st) {
    const int threads = 256;
    int64_t blocks = (r.total + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(splitk_reduce_set_kernel, dim3(static_cast<int>(blocks)), dim3(threads), 0, s,
                               r, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t splitk_reduce_launch(const float* part, float* y, int splits, int64_t count,
                                 cudaStream_t s, DevState st) {
    const int threads = 256;
    int64_t blocks = (count + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    cudaError_t e = launch_pdl(splitk_reduce_kernel, dim3(static_cast<int>(blocks)), dim3(threads), 0,
                               s, part, y, splits, count, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------ q8 quantizer
// One thread per 32-element block: amax, s = amax / 127 (IEEE fp32 division),
// x_q = round-half-even(x / s) clamped to [-127, 127]. A block whose scale is
// zero quantizes to zeros.

__device__ __forceinline__ void a16_store(uint16_t* a16, int64_t K, int64_t r, int64_t kb,
                                          const int (&q)[32]);

__global__ void quantize_q8_kernel(const void* __restrict__ x, int x_bf16, int64_t rows,
                                   int64_t K, int8_t* __restrict__ xq, float* __restrict__ xs,
                                   uint16_t* __restrict__ a16, int64_t rows_pad, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, 3);
    const int64_t nkb = K / 32;
    const int64_t nblk = rows_pad * nkb;
    for (int64_t blk = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; blk < nblk;
         blk += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = blk / nkb, kb = blk % nkb;
        int q[32];
        if (r < rows) {
            float v[32];
            load_x32(x, x_bf16, K, r, kb, v);
            const float s = quantize_block32(v, q);
            if (xq) {
                uint32_t pk[8];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    pk[m] = (q[4 * m] & 0xFF) | ((q[4 * m + 1] & 0xFF) << 8) |
                            ((q[4 * m + 2] & 0xFF) << 16) | ((q[4 * m + 3] & 0xFF) << 24);
                uint4* o = reinterpret_cast<uint4*>(xq + r * K + kb * 32);
                o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            xs[r * nkb + kb] = s;
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = 0;
        }
        if (a16) a16_store(a16, K, r, kb, q);
    }
}

// GEMM A-operand tile layout (must match gemm.cu): for every 128-row tile mt
// and every 32-column block kb, one 8 KB tile of fp16 values laid out as
// core matrices [row group rg (16)][k group kc (4)][row (8)][8 values].
__device__ __forceinline__ void a16_store(uint16_t* a16, int64_t K, int64_t r, int64_t kb,
                                          const int (&q)[32]) {
    const int64_t nkb = K / 32;
    const int64_t mt = r >> 7;
    const int rr = static_cast<int>(r & 127);
    uint16_t* tile = a16 + (mt * nkb + kb) * (128 * 32);
    const int rg = rr >> 3, rw = rr & 7;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = __half_as_ushort(__int2half_rn(q[8 * kc + 2 * j]));
            const uint32_t hi = __half_as_ushort(__int2half_rn(q[8 * kc + 2 * j + 1]));
            h[j] = lo | (hi << 16);
        }
        uint4* o = reinterpret_cast<uint4*>(tile + (rg * 4 + kc) * 64 + rw * 8);
        *o = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

cudaError_t quantize_q8_launch(const void* x, int x_bf16, int64_t rows, int64_t K, int8_t* xq,
                               float* xs, uint16_t* a16, cudaStream_t s, DevState st) {
    const int64_t rows_pad = a16 ? ((rows + 127) / 128) * 128 : rows;
    const int threads = 256;
    int64_t blocks = (rows_pad * (K / 32) + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    cudaError_t e = launch_pdl(quantize_q8_kernel, dim3(static_cast<int>(blocks)), dim3(threads), 0, s,
                               x, x_bf16, rows, K, xq, xs, a16, rows_pad, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------ W_exp plane
// plane[n][k] = q(n,k) - 32, one thread per 16-element group (16 ql bytes,
// 16 qh bytes, one shift pair), "57 - r54 MINFER_MMQ_Q6K_EXP" section 2.2.

__global__ void plane_build_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t K,
                                   int8_t* __restrict__ plane, DevState st) {
    live_bump(st, 4);
    const int64_t ngr = K / 16;
    const int64_t total = N * ngr;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = g / ngr, j = g % ngr;
        const int64_t sb = j / 16;
        const int e0 = static_cast<int>(j % 16) * 16;
        const uint8_t* blk = W + (n * (K / 256) + sb) * 210;
        const int s1 = 4 * (e0 >> 7), s2 = 2 * (e0 >> 6);
        uint32_t out[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t w = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int e = e0 + 4 * m + t;
                const int lo = (blk[e & 127] >> s1) & 0xF;
                const int hi = (blk[128 + (e & 63)] >> s2) & 0x3;
                w |= static_cast<uint32_t>(((lo | (hi << 4)) - 32) & 0xFF) << (8 * t);
            }
            out[m] = w;
        }
        *reinterpret_cast<uint4*>(plane + n * K + sb * 256 + e0) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

cudaError_t plane_build_launch(const uint8_t* W, int64_t N, int64_t K, int8_t* plane,
                               cudaStream_t s, DevState st) {
    const int threads = 256;
    int64_t blocks = (N * (K / 16) + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    plane_build_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(W, N, K, plane, st);
    return cudaGetLastError();
}

}  // namespace qmm
