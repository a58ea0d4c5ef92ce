// tcmv.cu -- host side of the tensor-core matvec (occupancy, launch) and the
// two small kernels that lay the activations out as its B operand.
#include <cuda_bf16.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "quant.cuh"
#include "tcmv.cuh"

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

// K offset within a 256-wide stage of the group with issue index i (the
// matvec issues a stage's groups quad by quad: q6_K quad Q holds the 16-wide
// groups Q, Q+4, Q+8, Q+12; Q4_0 / Q8_0 quad Q the 32-wide blocks 4Q..4Q+3)
__device__ __forceinline__ int group_k(int fmt, int i) {
    return fmt == FMT_Q6_K ? 16 * ((i >> 2) + 4 * (i & 3)) : 32 * i;
}

__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_val(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ float x_at(const void* x, int x_bf16, int64_t K, int b, int64_t k) {
    return x_bf16 ? bf16_val(static_cast<const uint16_t*>(x)[b * K + k])
                  : static_cast<const float*>(x)[b * K + k];
}

// The matvec's activation operand. Per 256-wide stage: 16 K16 steps t (group
// i = t / steps_per_group in issue order, half kk = t % steps_per_group), each
// an ncol x 16 bf16 matrix in core-matrix order [row / 8][k / 8][row % 8][k % 8].
// Row (i % G) * nc + c holds activation column c (batch row c / S, split
// c % S) at the group's K positions; all other rows are zero. Float mode: bf16
// activations as they are (S = 1) or fp32 ones split exactly as hi + mid + lo
// (S = 3). q8 mode: the per-32 int8 codes (exact in bf16), and the scales
// s[block][NB]. One thread per 16 bytes of the tile.
__device__ __forceinline__ void act_tile_unit(const void* __restrict__ x, int x_bf16, int B, int64_t K,
                                              int fmt, int NB, int S, int ncol, int q8,
                                              uint16_t* __restrict__ xt, float* __restrict__ xs, int64_t u) {
    const int nc = NB * S, G = ncol / nc;
    const int spg = fmt == FMT_Q6_K ? 1 : 2;  // K16 steps per group
    {
        // u enumerates [stage][t][row / 8][k8 (2)][row % 8]: consecutive
        // threads write consecutive 16-byte pieces
        const int r8 = static_cast<int>(u & 7);
        const int o = static_cast<int>((u >> 3) & 1);
        const int64_t rest = u >> 4;
        const int rg = static_cast<int>(rest % (ncol / 8));
        const int t = static_cast<int>((rest / (ncol / 8)) & 15);
        const int64_t stg = rest / (ncol / 8) / 16;
        const int r = rg * 8 + r8;
        const int i = t / spg, kk = t % spg;
        const int64_t k0 = stg * 256 + group_k(fmt, i) + 16 * kk + 8 * o;
        uint32_t h[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (r < G * nc && r / nc == i % G) {
            const int c = r % nc;
            const int b = c / S, j = c % S;
            if (q8) {
                // the 32-block of row b holding k0 (its 8 values are a quarter of it)
                const int64_t kb = k0 >> 5;
                float v[32];
                if (b < B && kb < K / 32)
                    load_x32(x, x_bf16, K, b, kb, v);
                else
                    for (int q = 0; q < 32; ++q) v[q] = 0.0f;
                int q[32];
                const float sc = quantize_block32(v, q);
                const int off = static_cast<int>(k0 & 31);
#pragma unroll
                for (int e = 0; e < 8; ++e) h[e] = bf16_bits(static_cast<float>(q[off + e]));
                if (off == 0) xs[kb * NB + b] = sc;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t k = k0 + e;
                    const float f = (b < B && k < K) ? x_at(x, x_bf16, K, b, k) : 0.0f;
                    if (S == 1) {
                        h[e] = bf16_bits(f);
                    } else {
                        // f = hi + mid + lo exactly (8 + 8 + 8 significant bits)
                        const uint32_t hi = bf16_bits(f);
                        const float r1 = f - bf16_val(hi);
                        const uint32_t mid = bf16_bits(r1);
                        const uint32_t lo = bf16_bits(r1 - bf16_val(mid));
                        h[e] = j == 0 ? hi : (j == 1 ? mid : lo);
                    }
                }
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(
            xt + stg * (static_cast<int64_t>(ncol) * 256) + static_cast<int64_t>(t) * ncol * 16 +
            (rg * 2 + o) * 64 + r8 * 8);
        *dst = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                          h[6] | (h[7] << 16));
    }
}

__global__ void act_tile_kernel(const void* __restrict__ x, int x_bf16, int B, int64_t K, int fmt,
                                int NB, int S, int ncol, int64_t nst, int q8,
                                uint16_t* __restrict__ xt, float* __restrict__ xs, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, q8 ? QMM_LIVE_QUANTIZE : QMM_LIVE_X_TILE);
    const int64_t units = nst * 16 * ncol * 2;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x)
        act_tile_unit(x, x_bf16, B, K, fmt, NB, S, ncol, q8, xt, xs, u);
}

// The same for the matrices of one grouped matvec in one launch: unit i
// belongs to the matrix m with start[m] <= i < start[m + 1].
__global__ void act_tile_set_kernel(const ActTileSet r, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, r.q8 ? QMM_LIVE_QUANTIZE : QMM_LIVE_X_TILE);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < r.total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int m = 0;
        for (int q = 1; q < r.n; ++q)
            if (i >= r.start[q]) m = q;
        act_tile_unit(r.x[m], r.x_bf16, r.B, r.K[m], r.fmt, r.NB, r.S, r.ncol, r.q8, r.xt[m], r.xs[m],
                      i - r.start[m]);
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

EncodeTiledFn tensor_map_encoder() {
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

namespace {

int row_slot_bytes(int fmt) { return fmt == FMT_Q6_K ? 240 : (fmt == FMT_Q4_0 ? 176 : 304); }

}  // namespace

namespace {

// W as [N / 8][8 * rowbytes] bytes of 16-bit elements: the pitch of 8 rows is
// a multiple of 16 bytes for every even row size; a box is one row slot wide
// and 16 groups of 8 rows high. No map (zeros) when W has fewer than 8 rows.
cudaError_t weight_map(int fmt, const TcmvArgs& a, CUtensorMap* map) {
    memset(map, 0, sizeof *map);
    if (a.n8 <= 0) return cudaSuccess;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(4 * a.rowbytes), static_cast<cuuint64_t>(a.n8 / 8)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(8 * a.rowbytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_slot_bytes(fmt) / 2), 16u};
    const cuuint32_t es[2] = {1u, 1u};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(a.W), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

}  // namespace

cudaError_t tcmv_launch_group(int fmt, bool q8, int NB, int S, int grid, cudaStream_t s, TcmvGroup& g) {
    TcmvKernel k = pick(fmt, q8, NB, S);
    if (!k || tcmv_occupancy(fmt, q8, NB, S) <= 0) return cudaErrorInvalidValue;
    if (g.nmat < 1 || g.nmat > kTcMaxMats) return cudaErrorInvalidValue;
    for (int m = 0; m < g.nmat; ++m) {
        cudaError_t e = weight_map(fmt, g.m[m], &g.map[m]);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(k, dim3(grid), dim3(kTcThreads), smem_of(fmt, NB, S), s, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t tcmv_launch(int fmt, bool q8, int NB, int S, int grid, cudaStream_t s,
                        const TcmvArgs& a) {
    static thread_local TcmvGroup g;  // large: kept off the stack
    g.nmat = 1;
    g.m[0] = a;
    g.m[0].item0 = 0;
    g.items = a.items;
    g.st = a.st;
    g.live_slot = a.live_slot;
    return tcmv_launch_group(fmt, q8, NB, S, grid, s, g);
}

cudaError_t act_tile_set_launch(const ActTileSet& r, cudaStream_t s, DevState st) {
    const int threads = 256;
    cudaError_t e = launch_pdl(act_tile_set_kernel, dim3(grid_for(r.total, threads)), dim3(threads), 0, s, r, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t act_tile_launch(const void* x, int x_bf16, int B, int64_t K, int fmt, int NB, int S,
                            int ncol, int64_t nst, bool q8, uint16_t* xt, float* xs, cudaStream_t s,
                            DevState st) {
    const int threads = 256;
    cudaError_t e = launch_pdl(act_tile_kernel, dim3(grid_for(nst * 16 * ncol * 2, threads)),
                               dim3(threads), 0, s, x, x_bf16, B, K, fmt, NB, S, ncol, nst,
                               q8 ? 1 : 0, xt, xs, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------ wait probe
// Test aid for the bounded waits: one warp waits, through the matvec's own
// warp-collective wait, on an mbarrier that nothing ever completes. After
// limit_ns of %globaltimer the wait gives up, raises the CTA's abort flag and
// the timeout bit of the error word, and the kernel returns. Nothing else is
// in flight in this kernel (no copies, no tensor memory), so the context
// stays usable and the next call runs normally.
__global__ void wait_probe_kernel(DevState st, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ uint32_t flag;
    const uint32_t b = smem_u32(&bar), f = smem_u32(&flag);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(f), "r"(0u) : "memory");
        fence_mbar_init();
    }
    __syncwarp();
    (void)tcmv_wait_warp(b, 0, f, st.err, limit_ns);
}

cudaError_t wait_probe_launch(unsigned long long limit_ns, cudaStream_t s, DevState st) {
    wait_probe_kernel<<<1, 32, 0, s>>>(st, limit_ns);
    return cudaGetLastError();
}

}  // namespace qmm
