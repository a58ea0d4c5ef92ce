// moe_prefill.cu -- the device steps of the expert-grouped MoE prefill
// (quantprobe "LAWS.md", L-30: prefill divides parameters rather than
// bytes, so a prompt's tokens are grouped by expert and each expert's
// weights are read once for all its tokens by the prefill GEMM):
//
//   plan:    the T*k routing slots ordered by expert, stable in slot order
//            (count per expert, then each expert's slots in slot order)
//   gather:  the activation row of each slot, in that order, so that an
//            expert's tokens are one contiguous GEMM input
//   silu:    h = silu(g) * u over the gate/up GEMM outputs, in place
//   combine: y[t] = sum_j gate[t][j] * o[pos(t, j)], in j order
//
// The GEMMs between them are the prefill GEMM's own launches (api.cu).
// Every step has a fixed order of operations, so results are bitwise
// reproducible.
#include <algorithm>

#include "kernels.h"

namespace qmm {

namespace {

constexpr int kPlanThreads = 256;

// one CTA per expert: its number of slots (slots outside 0..E-1 counted by
// CTA 0 as bad and flagged)
__global__ void __launch_bounds__(kPlanThreads) mp_count_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                               int* __restrict__ counts, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int e = static_cast<int>(blockIdx.x);
    int n = 0, bad = 0;
    for (int s = static_cast<int>(threadIdx.x); s < S; s += kPlanThreads) {
        const int v = __ldg(idx + s);
        n += v == e;
        bad += (v < 0 || v >= E);
    }
    __shared__ int red[kPlanThreads / 32][2];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        n += __shfl_xor_sync(0xffffffffu, n, o);
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[threadIdx.x >> 5][0] = n;
        red[threadIdx.x >> 5][1] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int tn = 0, tb = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            tn += red[w][0];
            tb += red[w][1];
        }
        counts[e] = tn;
        if (e == 0 && tb) atomicOr(st.err, DERR_MOE_BAD_INDEX);
    }
}

// one CTA per expert: its slots in slot order at its offset (the sum of the
// counts of the lower experts): order[off + r] = slot, pos[slot] = off + r
__global__ void __launch_bounds__(kPlanThreads) mp_order_kernel(const int32_t* __restrict__ idx, int S,
                                                               const int* __restrict__ counts,
                                                               int* __restrict__ order, int* __restrict__ pos,
                                                               DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_PLAN);
    const int e = static_cast<int>(blockIdx.x);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ int wsum[kPlanThreads / 32];
    __shared__ int base_s;
    // offset: the counts of experts 0 .. e-1
    int off = 0;
    for (int q = static_cast<int>(threadIdx.x); q < e; q += kPlanThreads) off += counts[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (lane == 0) wsum[warp] = off;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) t += wsum[w];
        base_s = t;
    }
    __syncthreads();
    int base = base_s;
    for (int s0 = 0; s0 < S; s0 += kPlanThreads) {
        const int s = s0 + static_cast<int>(threadIdx.x);
        const bool hit = s < S && __ldg(idx + s) == e;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        __syncthreads();  // wsum of the previous chunk has been read
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            before += w < warp ? wsum[w] : 0;
            total += wsum[w];
        }
        if (hit) {
            const int r = base + before + __popc(m & ((1u << lane) - 1u));
            order[r] = s;
            pos[s] = r;
        }
        base += total;
    }
}

// row r of Xg = the activation row of slot order[r] (token order[r] / k);
// rows of rowbytes (a multiple of 16) copied as 16-byte vectors
__global__ void __launch_bounds__(256) mp_gather_kernel(const uint8_t* __restrict__ x, int64_t rowbytes,
                                                       const int* __restrict__ order, int k, int S,
                                                       uint8_t* __restrict__ Xg, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_ROWS);
    const int64_t nv = rowbytes / 16;
    for (int r = static_cast<int>(blockIdx.x); r < S; r += static_cast<int>(gridDim.x)) {
        const int t = order[r] / k;
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * rowbytes);
        uint4* dst = reinterpret_cast<uint4*>(Xg + static_cast<int64_t>(r) * rowbytes);
        for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) dst[v] = __ldg(src + v);
    }
}

// The padded layout of the grouped launch: expert e's rows start at row
// poff[e] (a multiple of 128). pos_pad[s] = the slot's padded row, prow[row]
// = the slot of a padded row (left at -1 for padding rows).
__global__ void __launch_bounds__(256) mp_padmap_kernel(const int32_t* __restrict__ idx, const int* __restrict__ pos,
                                                       const int* __restrict__ off, const int* __restrict__ poff,
                                                       int S, int* __restrict__ pos_pad, int* __restrict__ prow,
                                                       DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_PLAN);
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < S; s += gridDim.x * blockDim.x) {
        const int e = idx[s];
        const int pp = poff[e] + (pos[s] - off[e]);
        pos_pad[s] = pp;
        prow[pp] = s;
    }
}

// padded row r of Xg = the activation row of slot prow[r], or zeros
__global__ void __launch_bounds__(256) mp_gather_pad_kernel(const uint8_t* __restrict__ x, int64_t rowbytes,
                                                           const int* __restrict__ prow, int k, int rows,
                                                           uint8_t* __restrict__ Xg, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_ROWS);
    const int64_t nv = rowbytes / 16;
    for (int r = static_cast<int>(blockIdx.x); r < rows; r += static_cast<int>(gridDim.x)) {
        const int s = prow[r];
        uint4* dst = reinterpret_cast<uint4*>(Xg + static_cast<int64_t>(r) * rowbytes);
        if (s < 0) {
            for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(s / k) * rowbytes);
            for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) dst[v] = __ldg(src + v);
        }
    }
}

// g <- silu(g) * u, element-wise over n values (n a multiple of 4)
__global__ void __launch_bounds__(256) mp_silu_kernel(float* __restrict__ g, const float* __restrict__ u,
                                                     int64_t n, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_SILU);
    const int64_t n4 = n / 4;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 a = reinterpret_cast<float4*>(g)[i];
        const float4 b = __ldg(reinterpret_cast<const float4*>(u) + i);
        a.x = a.x / (1.0f + expf(-a.x)) * b.x;
        a.y = a.y / (1.0f + expf(-a.y)) * b.y;
        a.z = a.z / (1.0f + expf(-a.z)) * b.z;
        a.w = a.w / (1.0f + expf(-a.w)) * b.w;
        reinterpret_cast<float4*>(g)[i] = a;
    }
}

// y[t][n] = sum_j gate[t*k + j] * O[pos[t*k + j]][n], j in order; blockIdx.x
// = token, threads over n in float4 (H a multiple of 4)
__global__ void __launch_bounds__(256) mp_combine_kernel(const float* __restrict__ O, const int* __restrict__ pos,
                                                        const float* __restrict__ gate, int k, int H,
                                                        float* __restrict__ y, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_PREFILL_ROWS);
    const int t = static_cast<int>(blockIdx.x);
    const int h4 = H / 4;
    for (int v = static_cast<int>(threadIdx.x); v < h4; v += static_cast<int>(blockDim.x)) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int j = 0; j < k; ++j) {
            const float gw = gate[t * k + j];
            const float4 o = __ldg(reinterpret_cast<const float4*>(O + static_cast<int64_t>(pos[t * k + j]) * H) + v);
            acc.x = fmaf(gw, o.x, acc.x);
            acc.y = fmaf(gw, o.y, acc.y);
            acc.z = fmaf(gw, o.z, acc.z);
            acc.w = fmaf(gw, o.w, acc.w);
        }
        reinterpret_cast<float4*>(y + static_cast<int64_t>(t) * H)[v] = acc;
    }
}

}  // namespace

cudaError_t moe_prefill_plan_launch(const int32_t* idx, int S, int E, int* counts, int* order, int* pos,
                                    cudaStream_t s, DevState st) {
    cudaError_t e = launch_pdl(mp_count_kernel, dim3(static_cast<unsigned>(E)), dim3(kPlanThreads), 0, s, idx, S, E,
                               counts, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(mp_order_kernel, dim3(static_cast<unsigned>(E)), dim3(kPlanThreads), 0, s, idx, S,
                      static_cast<const int*>(counts), order, pos, st);
}

cudaError_t moe_prefill_gather_launch(const void* x, int64_t rowbytes, const int* order, int k, int S, void* Xg,
                                      int sms, cudaStream_t s, DevState st) {
    const int grid = static_cast<int>(std::min<int64_t>(S, static_cast<int64_t>(sms) * 8));
    return launch_pdl(mp_gather_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                      static_cast<const uint8_t*>(x), rowbytes, order, k, S, static_cast<uint8_t*>(Xg), st);
}

cudaError_t moe_prefill_padmap_launch(const int32_t* idx, const int* pos, const int* off, const int* poff, int S,
                                      int* pos_pad, int* prow, int sms, cudaStream_t s, DevState st) {
    const int blocks = std::max(1, std::min((S + 255) / 256, sms * 4));
    return launch_pdl(mp_padmap_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, idx, pos, off, poff, S,
                      pos_pad, prow, st);
}

cudaError_t moe_prefill_gather_pad_launch(const void* x, int64_t rowbytes, const int* prow, int k, int rows, void* Xg,
                                          int sms, cudaStream_t s, DevState st) {
    const int grid = static_cast<int>(std::min<int64_t>(rows, static_cast<int64_t>(sms) * 8));
    return launch_pdl(mp_gather_pad_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                      static_cast<const uint8_t*>(x), rowbytes, prow, k, rows, static_cast<uint8_t*>(Xg), st);
}

cudaError_t moe_prefill_silu_launch(float* g, const float* u, int64_t n, int sms, cudaStream_t s, DevState st) {
    const int64_t blocks = std::min<int64_t>((n / 4 + 255) / 256, static_cast<int64_t>(sms) * 8);
    return launch_pdl(mp_silu_kernel, dim3(static_cast<unsigned>(std::max<int64_t>(blocks, 1))), dim3(256), 0, s, g,
                      u, n, st);
}

cudaError_t moe_prefill_combine_launch(const float* O, const int* pos, const float* gate, int T, int k, int H,
                                       float* y, cudaStream_t s, DevState st) {
    return launch_pdl(mp_combine_kernel, dim3(static_cast<unsigned>(T)), dim3(256), 0, s, O, pos, gate, k, H, y, st);
}

}  // namespace qmm
