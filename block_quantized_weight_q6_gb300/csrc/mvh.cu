// mvh.cu -- host side of the batch 1-8 fp16-MMA matvec (mvh.cuh): the
// activation prep kernel, the weight tensor maps, the team size and the launch.
#include <string.h>

#include <algorithm>
#include <mutex>

#include "mvh.cuh"

namespace qmm {

// ------------------------------------------------------------ prep
// One CTA per (distinct activation matrix, batch row): the row's largest
// magnitude fixes e (largest value times 2^e in [2^14, 2^15)), then every
// value is written as fp16 x * 2^e (exact for bf16 values within 2^28 of the
// largest), and 2^-e is kept for the output.
constexpr int kPrepMax = kMvhMaxMats;
struct MvhPrep {
    const uint16_t* x[kPrepMax];
    uint16_t* xh[kPrepMax];
    float* xinv[kPrepMax];
    int64_t K[kPrepMax];
    int* ctr;  // the matvec's item counter, reset here
    int n, B;
};

__global__ void __launch_bounds__(256) mvh_prep_kernel(const __grid_constant__ MvhPrep p, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();  // x comes from the previous kernel, which no longer uses the counter
    live_bump(st, QMM_LIVE_X_TILE);
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.ctr = 0;
    const int i = blockIdx.x / p.B, b = blockIdx.x % p.B;
    const int64_t K = p.K[i];
    const uint16_t* x = p.x[i] + static_cast<int64_t>(b) * K;
    uint16_t* xh = p.xh[i] + static_cast<int64_t>(b) * K;
    // magnitude bits of bf16 order like the magnitudes (NaN above infinity)
    uint32_t mb = 0;
    for (int64_t k = 8 * static_cast<int64_t>(threadIdx.x); k < K; k += 8 * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) mb = max(mb, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mb;
    __syncthreads();
    mb = red[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) mb = max(mb, red[w]);
    int s = 0;
    if (mb != 0 && mb < 0x7F80u) {  // finite and nonzero
        int e;
        (void)frexpf(__uint_as_float(mb << 16), &e);  // largest magnitude < 2^e
        s = min(126, max(-126, 15 - e));  // 2^s and 2^-s stay normal fp32 numbers
    }
    const float sc = ldexpf(1.0f, s);
    for (int64_t k = 8 * static_cast<int64_t>(threadIdx.x); k < K; k += 8 * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half lo = __float2half_rn(__uint_as_float(w[q] << 16) * sc);
            const __half hi = __float2half_rn(__uint_as_float(w[q] & 0xFFFF0000u) * sc);
            o[q] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
        }
        *reinterpret_cast<uint4*>(xh + k) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (threadIdx.x == 0) p.xinv[i][b] = ldexpf(1.0f, -s);
}

// ------------------------------------------------------------ host

bool mvh_supported(int fmt, int64_t N, int64_t K) {
    return (fmt == FMT_Q4_0 || fmt == FMT_Q8_0 || fmt == FMT_Q6_K) && K > 0 && K % 256 == 0 && N >= 8 &&
           N % 8 == 0 && N / 8 <= (int64_t{1} << 31) - 1;
}

namespace {

size_t round256(size_t v) { return (v + 255) / 256 * 256; }
int block_elems(int f) { return f == FMT_Q6_K ? 256 : 32; }
int block_bytes(int f) { return f == FMT_Q6_K ? 210 : (f == FMT_Q4_0 ? 18 : 34); }

// distinct activation matrices among x[0 .. n-1] (same pointer and K): their
// index for each matrix and their workspace offsets
struct XPlan {
    int which[kMvhMaxMats];
    int nd;
    const void* x[kMvhMaxMats];
    int64_t K[kMvhMaxMats];
    size_t xh_off[kMvhMaxMats], xinv_off[kMvhMaxMats], total;
};

void plan_x(int n, const void* const* x, const int64_t* K, int B, XPlan* p) {
    p->nd = 0;
    p->total = 256;  // the item counter
    for (int i = 0; i < n; ++i) {
        int d = -1;
        for (int q = 0; q < p->nd; ++q)
            if (p->x[q] == x[i] && p->K[q] == K[i]) d = q;
        if (d < 0) {
            d = p->nd++;
            p->x[d] = x[i];
            p->K[d] = K[i];
            p->xh_off[d] = p->total;
            p->total = round256(p->total + static_cast<size_t>(B) * K[i] * 2);
            p->xinv_off[d] = p->total;
            p->total = round256(p->total + static_cast<size_t>(B) * 4);
        }
        p->which[i] = d;
    }
}

cudaError_t prepare_kernel() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(mvh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kMvhSmem));
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(mvh_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
    });
    return err;
}

}  // namespace

size_t mvh_workspace_bytes(int n, const void* const* x, const int64_t* K, int B) {
    if (n < 1 || n > kMvhMaxMats) return 0;
    XPlan p;
    plan_x(n, x, K, B, &p);
    return p.total;
}

cudaError_t mvh_run(int n, const int* sel, const int* fmt, const void* const* W, const void* const* x,
                    float* const* y, const int64_t* N, const int64_t* K, int B, void* ws, int sms,
                    cudaStream_t s, DevState st) {
    if (n < 1 || n > kMvhMaxMats || B < 1 || B > 8) return cudaErrorInvalidValue;
    cudaError_t e = prepare_kernel();
    if (e != cudaSuccess) return e;
    // matrices in order of stages per item, longest first: the round-robin
    // walk of the items then starts the long ones first
    int ord[kMvhMaxMats];
    for (int i = 0; i < n; ++i) ord[i] = sel[i];
    auto stages_of = [&](int m) { return K[m] / (fmt[m] == FMT_Q8_0 ? 128 : 256); };
    std::stable_sort(ord, ord + n, [&](int a, int b) { return stages_of(a) > stages_of(b); });
    const void* xs[kMvhMaxMats];
    int64_t Ks[kMvhMaxMats];
    for (int i = 0; i < n; ++i) {
        xs[i] = x[ord[i]];
        Ks[i] = K[ord[i]];
    }
    XPlan xp;
    plan_x(n, xs, Ks, B, &xp);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    MvhPrep pr{};
    pr.ctr = reinterpret_cast<int*>(wsb);
    pr.n = xp.nd;
    pr.B = B;
    for (int d = 0; d < xp.nd; ++d) {
        pr.x[d] = static_cast<const uint16_t*>(xp.x[d]);
        pr.xh[d] = reinterpret_cast<uint16_t*>(wsb + xp.xh_off[d]);
        pr.xinv[d] = reinterpret_cast<float*>(wsb + xp.xinv_off[d]);
        pr.K[d] = xp.K[d];
    }
    e = launch_pdl(mvh_prep_kernel, dim3(static_cast<unsigned>(xp.nd * B)), dim3(256), 0, s, pr, st);
    if (e != cudaSuccess) return e;

    static thread_local MvhGroup g;  // large: kept off the stack
    memset(&g, 0, sizeof g);
    g.nmat = n;
    g.ctr = pr.ctr;
    g.B = B;
    g.st = st;
    g.live_slot = QMM_LIVE_GEMV_MV8;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    int64_t items = 0;
    int min_stages = 1 << 30;
    for (int i = 0; i < n; ++i) {
        const int m = ord[i];
        MvhMat& a = g.m[i];
        a.W = static_cast<const uint8_t*>(W[m]);
        a.xh = pr.xh[xp.which[i]];
        a.xinv = pr.xinv[xp.which[i]];
        a.y = y[m];
        a.N = N[m];
        a.K = K[m];
        a.fmt = fmt[m];
        a.rowbytes = K[m] / block_elems(a.fmt) * block_bytes(a.fmt);
        a.stages = static_cast<int>(K[m] / (a.fmt == FMT_Q8_0 ? 128 : 256));
        a.item0 = static_cast<int>(items);
        items += (N[m] + 8 * kMvhRows - 1) / (8 * kMvhRows) * 8;
        min_stages = std::min(min_stages, a.stages);
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(4 * a.rowbytes), static_cast<cuuint64_t>(N[m] / 8)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(8 * a.rowbytes)};
        const cuuint32_t box[2] = {mvh_box_w(a.fmt) / 2, static_cast<cuuint32_t>(kMvhRows)};
        const cuuint32_t es[2] = {1u, 1u};
        if (enc(&g.map[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(a.W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (items > (int64_t{1} << 30)) return cudaErrorInvalidValue;
    g.items = static_cast<int>(items);
    // warps per item: enough that the items keep every warp of the grid
    // busy, at most any matrix's stages
    const int64_t warps = static_cast<int64_t>(sms) * kMvhWarps;
    // (a divisor of the CTA's warps: teams never span two CTAs)
    g.ks = 1;
    for (int k : {1, 2, 4, 8, 16}) {
        if (k > min_stages) break;
        g.ks = k;
        if (items * k >= warps) break;
    }
    const int64_t per_cta = kMvhWarps / g.ks;
    const int grid = static_cast<int>(std::min<int64_t>(sms, (items + per_cta - 1) / per_cta));
    e = launch_pdl(mvh_kernel, dim3(grid), dim3(kMvhWarps * 32), kMvhSmem, s, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmm
