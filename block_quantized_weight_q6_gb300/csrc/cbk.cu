// cbk.cu -- matvec against an additive-codebook matrix ("Chasing x100",
// "The kernel is ready": the 2-bit / 3-bit additive codebook matvec):
//
//   w[n][8g + j] = scale[n] * sum_m books[m][codes[n][g][m]][j]
//   y[b][n]      = sum_k w[n][k] * x[b][k]
//
// M = 2 or 3 books of 256 fp16 8-vectors, one code byte per book per 8
// weights (2 or 3 bits per weight). A matvec over such a matrix reads one
// byte per book and group, so its work is a table lookup, not a decode:
// the dot of every book entry with each 8-wide slice of the activations,
//   T[b][m][c][g] = sum_j books[m][c][j] * x[b][8g + j]   (fp32, j in order),
// is built once per CTA for its chunk of G groups and shared by all the
// rows the CTA walks; a row's sum over the chunk is then M lookups per group
// and batch row. Lanes take consecutive groups of one row, so the table is
// laid out with g fastest and one warp-wide lookup reads G different
// columns (32 / G rows per warp). The partial sums of the
// chunks are added in chunk order by a second launch, which applies the row
// scale, so results do not depend on timing.
#include <algorithm>

#include "kernels.h"

namespace qmm {

namespace {

constexpr int kCbkThreads = 256;
// rows whose codes are staged at a time (double-buffered)
template <int G>
__host__ __device__ constexpr int cbk_row_block() { return G == 16 ? 256 : 128; }

__device__ __forceinline__ void cbk_cp8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cbk_cp16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cbk_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cbk_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The codes of rows n0 .. n0 + rows - 1 for the chunk's groups (G * M bytes
// a row, 8-byte pieces) into cs.
template <int M, int G>
__device__ __forceinline__ void cbk_stage(const uint8_t* codes, int64_t ng, int64_t g0, int64_t n0, int rows,
                                          uint8_t* cs) {
    constexpr int kPieces = G * M / 8;
    const uint32_t base = smem_u32(cs);
    for (int i = static_cast<int>(threadIdx.x); i < rows * kPieces; i += kCbkThreads) {
        const int r = i / kPieces, q = i % kPieces;
        cbk_cp8(base + static_cast<uint32_t>(r * G * M + 8 * q), codes + ((n0 + r) * ng + g0) * M + 8 * q);
    }
}

template <int M, int G, int NB>
__global__ void __launch_bounds__(kCbkThreads) cbk_kernel(const uint8_t* __restrict__ codes,
                                                         const uint16_t* __restrict__ books,
                                                         const void* __restrict__ x, int x_bf16, int64_t N,
                                                         int64_t K, int B, int64_t rows_per_slice,
                                                         float* __restrict__ part, DevState st) {
    extern __shared__ __align__(16) float sm[];
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_CBK_GEMV);
    const int chunk = static_cast<int>(blockIdx.x);
    const int64_t g0 = static_cast<int64_t>(chunk) * G;
    const int64_t ng = K / 8;
    const int64_t n_lo = static_cast<int64_t>(blockIdx.y) * rows_per_slice;
    const int64_t n_hi = n_lo + rows_per_slice < N ? n_lo + rows_per_slice : N;
    float* xs = sm;                                      // [B][8G] activations of the chunk
    float* bs = xs + static_cast<size_t>(B) * 8 * G;     // [M][256][8] the books as fp32
    float* T = bs + static_cast<size_t>(M) * 256 * 8;    // [B][M][256][G]
    uint8_t* cs = reinterpret_cast<uint8_t*>(T + static_cast<size_t>(B) * M * 256 * G);  // [2][block][G * M]
    constexpr int kCbkRowBlock = cbk_row_block<G>();
    constexpr int kCsBuf = kCbkRowBlock * G * M;
    // the first block of codes, the books (fp16) and the chunk's activations
    // travel together; the raw books and activations land in the table's
    // space, which is built only after they are converted
    const int nblocks = static_cast<int>((n_hi - n_lo + kCbkRowBlock - 1) / kCbkRowBlock);
    if (nblocks > 0) {
        cbk_stage<M, G>(codes, ng, g0, n_lo, static_cast<int>(n_hi - n_lo < kCbkRowBlock ? n_hi - n_lo : kCbkRowBlock),
                        cs);
    }
    uint8_t* raw = reinterpret_cast<uint8_t*>(T);
    constexpr int kBookBytes = M * 256 * 8 * 2;
    const int xb = x_bf16 ? 2 : 4;
    const int xrow = 8 * G * xb;  // bytes of a batch row's chunk
    {
        const uint32_t rb = smem_u32(raw);
        for (int i = static_cast<int>(threadIdx.x); i < kBookBytes / 16; i += kCbkThreads)
            cbk_cp16(rb + 16 * i, reinterpret_cast<const uint8_t*>(books) + 16 * i);
        for (int i = static_cast<int>(threadIdx.x); i < B * xrow / 16; i += kCbkThreads) {
            const int b = i / (xrow / 16), q = i % (xrow / 16);
            cbk_cp16(rb + kBookBytes + 16 * i,
                     static_cast<const uint8_t*>(x) + (b * K + 8 * g0) * xb + 16 * q);
        }
    }
    cbk_commit();
    cbk_wait<0>();
    __syncthreads();
    {
        const uint16_t* rbk = reinterpret_cast<const uint16_t*>(raw);
        for (int i = static_cast<int>(threadIdx.x); i < M * 256 * 8; i += kCbkThreads)
            bs[i] = __half2float(__ushort_as_half(rbk[i]));
        const uint8_t* rx = raw + kBookBytes;
        for (int i = static_cast<int>(threadIdx.x); i < B * 8 * G; i += kCbkThreads)
            xs[i] = x_bf16 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rx)[i]) << 16)
                           : reinterpret_cast<const float*>(rx)[i];
    }
    __syncthreads();  // the raw copies are read before the table overwrites them
    // the table: thread (c0, g) takes entries c = c0, c0 + 256 / G, ... of
    // group g, its 8 activations in registers (consecutive threads write
    // consecutive words; the 32 / G threads of one c read one book entry)
    {
        constexpr int kCStep = kCbkThreads / G;
        const int g = static_cast<int>(threadIdx.x) % G, c0 = static_cast<int>(threadIdx.x) / G;
        for (int b = 0; b < B; ++b) {
            const float4 x0 = reinterpret_cast<const float4*>(xs + b * 8 * G + 8 * g)[0];
            const float4 x1 = reinterpret_cast<const float4*>(xs + b * 8 * G + 8 * g)[1];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float* Tm = T + (static_cast<size_t>(b) * M + m) * 256 * G;
                const float* bm = bs + m * 256 * 8;
#pragma unroll 4
                for (int c = c0; c < 256; c += kCStep) {
                    const float4 e0 = reinterpret_cast<const float4*>(bm + c * 8)[0];
                    const float4 e1 = reinterpret_cast<const float4*>(bm + c * 8)[1];
                    float p = 0.0f;
                    p = fmaf(e0.x, x0.x, p);
                    p = fmaf(e0.y, x0.y, p);
                    p = fmaf(e0.z, x0.z, p);
                    p = fmaf(e0.w, x0.w, p);
                    p = fmaf(e1.x, x1.x, p);
                    p = fmaf(e1.y, x1.y, p);
                    p = fmaf(e1.z, x1.z, p);
                    p = fmaf(e1.w, x1.w, p);
                    Tm[c * G + g] = p;
                }
            }
        }
    }
    // rows: a warp takes 32 / G rows at a time, lane = (row r, group g)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRpw = 32 / G;
    const int r = lane / G, g = lane % G;
    for (int blk = 0; blk < nblocks; ++blk) {
        const int64_t nb0 = n_lo + static_cast<int64_t>(blk) * kCbkRowBlock;
        const int rows = static_cast<int>(n_hi - nb0 < kCbkRowBlock ? n_hi - nb0 : kCbkRowBlock);
        // the next block's codes go out before this one is used
        if (blk + 1 < nblocks) {
            const int64_t nn = nb0 + kCbkRowBlock;
            cbk_stage<M, G>(codes, ng, g0, nn,
                            static_cast<int>(n_hi - nn < kCbkRowBlock ? n_hi - nn : kCbkRowBlock),
                            cs + ((blk + 1) & 1) * kCsBuf);
        }
        cbk_commit();
        cbk_wait<1>();
        __syncthreads();  // the block's codes (and, the first time, the table) are in place
        const uint8_t* cb = cs + (blk & 1) * kCsBuf;
        for (int rb = warp * kRpw; rb < rows; rb += (kCbkThreads / 32) * kRpw) {
            const int rr = rb + r;
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
            if (rr < rows) {
                const uint8_t* cp = cb + rr * G * M + g * M;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int c = cp[m];
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        if (NB == 1 || b < B) acc[b] += T[((b * M + m) * 256 + c) * G + g];
                }
            }
            // the row's sum over its G lanes, in a fixed tree order
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (NB > 1 && b >= B) break;
                float v = acc[b];
#pragma unroll
                for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (g == 0 && rr < rows) part[(static_cast<int64_t>(chunk) * B + b) * N + nb0 + rr] = v;
            }
        }
        __syncthreads();  // this buffer is refilled two blocks on
    }
    cbk_wait<0>();
}

// y[b][n] = scale[n] * sum_chunk part[chunk][b][n], chunks in order
__global__ void __launch_bounds__(256) cbk_reduce_kernel(const float* __restrict__ part,
                                                        const uint16_t* __restrict__ scales, int chunks, int B,
                                                        int64_t N, float* __restrict__ y, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_CBK_GEMV);
    const int64_t total = static_cast<int64_t>(B) * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i % N;
        float s = 0.0f;
        for (int c = 0; c < chunks; ++c) s += part[static_cast<int64_t>(c) * total + i];
        y[i] = __half2float(__ushort_as_half(scales[n])) * s;
    }
}

}  // namespace

// groups per chunk: 16, or 8 where the table would not fit
int cbk_group_width(int M, int B) { return B * M <= 8 ? 16 : 8; }

size_t cbk_smem_bytes(int M, int B) {
    const int G = cbk_group_width(M, B);
    const int rb = G == 16 ? cbk_row_block<16>() : cbk_row_block<8>();
    return static_cast<size_t>(B) * 8 * G * 4 + static_cast<size_t>(M) * 256 * 8 * 4 +
           static_cast<size_t>(B) * M * 256 * G * 4 + 2 * static_cast<size_t>(rb) * G * M;
}

int cbk_chunks(int64_t K, int M, int B) {
    const int64_t G = cbk_group_width(M, B);
    return static_cast<int>((K / 8 + G - 1) / G);
}

size_t cbk_part_bytes(int M, int64_t N, int64_t K, int B) {
    return static_cast<size_t>(cbk_chunks(K, M, B)) * B * N * 4;
}

cudaError_t cbk_launch(int M, const uint8_t* codes, const uint16_t* books, const uint16_t* scales, const void* x,
                       int x_bf16, float* y, int64_t N, int64_t K, int B, float* part, int sms, cudaStream_t s,
                       DevState st) {
    const int G = cbk_group_width(M, B);
    const int chunks = cbk_chunks(K, M, B);
    const size_t smem = cbk_smem_bytes(M, B);
    // row slices: enough CTAs for four per SM, a slice at least 256 rows
    int64_t slices = std::max<int64_t>(1, (4 * static_cast<int64_t>(sms) + chunks - 1) / chunks);
    slices = std::min<int64_t>(slices, std::max<int64_t>(1, N / 256));
    const int64_t rps = (N + slices - 1) / slices;
    if (chunks > 65535 || slices > 65535) return cudaErrorInvalidValue;
    // batch width instantiations: 1, 2, 4, 8 rows (the chunk width follows
    // B * M, so only these pairs occur)
    using Kern = void (*)(const uint8_t*, const uint16_t*, const void*, int, int64_t, int64_t, int, int64_t, float*,
                          DevState);
    Kern kern;
    const int nb = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
    if (M == 2) {
        kern = nb == 1 ? cbk_kernel<2, 16, 1> : nb == 2 ? cbk_kernel<2, 16, 2> : nb == 4 ? cbk_kernel<2, 16, 4>
                                                                                       : cbk_kernel<2, 8, 8>;
    } else {
        kern = nb == 1 ? cbk_kernel<3, 16, 1> : nb == 2 ? cbk_kernel<3, 16, 2> : nb == 4 ? cbk_kernel<3, 8, 4>
                                                                                       : cbk_kernel<3, 8, 8>;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(slices)), dim3(kCbkThreads), smem,
                   s, codes, books, x, x_bf16, N, K, B, rps, part, st);
    if (e != cudaSuccess) return e;
    const int64_t blocks = std::min<int64_t>((static_cast<int64_t>(B) * N + 255) / 256, static_cast<int64_t>(sms) * 8);
    return launch_pdl(cbk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                      static_cast<const float*>(part), scales, chunks, B, N, y, st);
}

}  // namespace qmm
