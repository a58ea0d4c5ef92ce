// gemv.cu -- host-side dispatch of the matvec kernels (their device code is
// in gemv_impl.cuh, instantiated per format), and the small kernels around
// them: the per-32 activation quantizer, the bf16 -> fp32 activation copy,
// the split-K reduction and the W_exp plane build.
#include <map>
#include <mutex>
#include <utility>

#include "gemv_impl.cuh"

namespace qmm {

// ------------------------------------------------------------ dispatch

size_t gemv_smem_bytes(int fmt, int R) {
    const int seg = fmt == FMT_Q6_K ? seg_stride<FMT_Q6_K>()
                                    : (fmt == FMT_Q4_0 ? seg_stride<FMT_Q4_0>() : seg_stride<FMT_Q8_0>());
    const int ns = R >= 4 ? slots_for<4>() : (R == 2 ? slots_for<2>() : slots_for<1>());
    return static_cast<size_t>(kGemvWarps) * ns * seg * R + kGemvWarps * ns * 8;
}

int gemv_chunk_blocks(int fmt) {
    return fmt == FMT_Q6_K ? Fmt<FMT_Q6_K>::CB : Fmt<FMT_Q4_0>::CB;
}

static GemvKernel pick_kernel(int fmt, bool q8, int NB, int R) {
    switch (fmt) {
    case FMT_Q6_K: return gemv_pick_q6k(q8, NB, R);
    case FMT_Q4_0: return gemv_pick_q4_0(q8, NB, R);
    case FMT_Q8_0: return gemv_pick_q8_0(q8, NB, R);
    }
    return nullptr;
}

// Sets the kernel's shared-memory opt-in and returns its resident CTAs per SM;
// both are computed once per (kernel, device) and cached.
int gemv_occupancy(int fmt, bool q8, int NB, int R) {
    GemvKernel k = pick_kernel(fmt, q8, NB, R);
    if (!k) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    static std::mutex mu;
    static std::map<std::pair<int, GemvKernel>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, k});
    if (it != cache.end()) return it->second;
    const size_t smem = gemv_smem_bytes(fmt, R);
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kGemvThreads, smem) != cudaSuccess)
        n = 0;
    cache[{dev, k}] = n;
    return n;
}

cudaError_t gemv_launch(int fmt, bool q8, int NB, int R, int grid, cudaStream_t s,
                        const GemvArgs& a) {
    GemvKernel k = pick_kernel(fmt, q8, NB, R);
    if (!k) return cudaErrorInvalidValue;
    const size_t smem = gemv_smem_bytes(fmt, R);
    // the shared-memory opt-in is set once per kernel (gemv_occupancy, called
    // by the planner before the first launch), so that a launch inside a
    // stream capture issues nothing but the launch itself
    if (gemv_occupancy(fmt, q8, NB, R) <= 0) return cudaErrorInvalidConfiguration;
    cudaError_t e = launch_pdl(k, dim3(grid), dim3(kGemvThreads), smem, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------ bf16 -> fp32

__global__ void x_to_f32_kernel(const uint16_t* __restrict__ x, float* __restrict__ o, int64_t n,
                                DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_X_WIDEN);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        o[i] = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
}

cudaError_t x_to_f32_launch(const void* x_bf16, float* out, int64_t n, cudaStream_t s,
                            DevState st) {
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    cudaError_t e = launch_pdl(x_to_f32_kernel, dim3(static_cast<int>(blocks)), dim3(threads), 0, s,
                               static_cast<const uint16_t*>(x_bf16), out, n, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

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
            if (x_bf16) {
                const uint4* p = reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(x) + r * K + kb * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 u = __ldg(p + i);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                        v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                    }
                }
            } else {
                const float4* p =
                    reinterpret_cast<const float4*>(static_cast<const float*>(x) + r * K + kb * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 u = __ldg(p + i);
                    v[4 * i] = u.x;
                    v[4 * i + 1] = u.y;
                    v[4 * i + 2] = u.z;
                    v[4 * i + 3] = u.w;
                }
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
            const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                int t = 0;
                if (s != 0.0f) {
                    t = __float2int_rn(__fdiv_rn(v[i], s));
                    t = max(-127, min(127, t));
                }
                q[i] = t;
            }
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
