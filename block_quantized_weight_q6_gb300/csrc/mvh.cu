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
    return (fmt == FMT_Q4_0 || fmt == FMT_Q8_0 || fmt == FMT_Q6_K || fmt == FMT_Q4_K || fmt == FMT_Q2_K) && K > 0 &&
           K % 256 == 0 && N >= 8 &&
           N % 8 == 0 && N / 8 <= (int64_t{1} << 31) - 1;
}

namespace {

size_t round256(size_t v) { return (v + 255) / 256 * 256; }
int block_elems(int f) { return (f == FMT_Q4_0 || f == FMT_Q8_0) ? 32 : 256; }
int block_bytes(int f) {
    return f == FMT_Q6_K ? 210 : f == FMT_Q4_0 ? 18 : f == FMT_Q8_0 ? 34 : f == FMT_Q4_K ? 144 : 84;
}

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
        for (auto k : {mvh_kernel<false>, mvh_kernel<true>}) {
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMvhSmem));
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
        }
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
        a.stage_bytes = mvh_stage_bytes(a.fmt);
        a.stage_k = mvh_stage_k(a.fmt);
        a.box_w = static_cast<int>(mvh_box_w(a.fmt));
        a.boxes = mvh_boxes(a.fmt);
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
    bool kq = false;
    for (int i = 0; i < n; ++i) kq = kq || fmt[ord[i]] == FMT_Q4_K || fmt[ord[i]] == FMT_Q2_K;
    e = launch_pdl(kq ? mvh_kernel<true> : mvh_kernel<false>, dim3(grid), dim3(kMvhWarps * 32), kMvhSmem, s, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ================================================================ routed experts
// The expert matvecs of moe_gemv on the same stages and tiles. An item is
// (task, matrix of the launch, 16-row block at stride 8); the task gives the
// expert (the third coordinate of the table's tensor map), the task's first
// grouped slot and its tokens. gate/up launch: two matrices, B = tokens, each
// token's activations one fp16 row (scaled per slot). down launch: one
// matrix, each token's h as two fp16 rows hi + lo (22 bits of its fp32
// value), B = 2 tokens, and a token's output is the sum of its two columns.
struct MvhMoeArgs {
    CUtensorMap map[2];      // W as [E][N / 8][8 * rowbytes] 16-bit elements
    const int* n_tasks;
    const MoeTask* tasks;
    const uint16_t* xh;      // fp16 activation rows (slot, or 2 slot + part)
    const float* xinv;       // [slots] 2^-e of each slot's rows
    float* out[2];           // [slots][N]
    int64_t N, K, rowbytes;
    int nmat, split, ks;
    int* ctr;
    DevState st;
    int live_slot;
};

template <int FMT>
__global__ void __launch_bounds__(kMvhWarps * 32, 1) moe_mvh_kernel(const __grid_constant__ MvhMoeArgs g) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, c = lane & 3;
    const int ks = g.ks;
    const int team = warp / ks, member = warp % ks;
    const uint32_t S = smem_u32(smem);
    const uint32_t ring = S + static_cast<uint32_t>(warp) * kMvhNS * kMvhSlot;
    const uint32_t bars = S + kMvhBarOff + static_cast<uint32_t>(warp) * kMvhNS * 8;
    float* part = reinterpret_cast<float*>(smem + kMvhPartOff);
    int* fifo = reinterpret_cast<int*>(smem + kMvhFifoOff) + 4 * warp;
    const int nteams = static_cast<int>(gridDim.x) * (kMvhWarps / ks);
    const int gt = team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    const uint32_t selc = 0x4040u | (static_cast<uint32_t>(c) << 8) | static_cast<uint32_t>(c);
    Q6Off po;
    po.o[0] = q6k_poff(c);
    po.o[1] = q6k_poff(c + 1);
    po.o[2] = q6k_poff(4 + c);
    po.o[3] = q6k_poff(5 + c);
    po.o[4] = q6k_poff(8 + c);
    po.o[5] = q6k_poff(9 + c);
    constexpr int SB = mvh_stage_bytes(FMT), SK = mvh_stage_k(FMT);
    constexpr int NBX = mvh_boxes(FMT);
    constexpr uint32_t BW = mvh_box_w(FMT);
    const int stages = static_cast<int>(g.K / SK);
    const int ipm = static_cast<int>((g.N + 8 * kMvhRows - 1) / (8 * kMvhRows)) * 8;  // items per matrix

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (lane < kMvhNS) mbar_init(bars + 8 * lane, 1);
    fence_mbar_init();
    __syncwarp();
    // the tasks, the activations and the counter come from earlier kernels
    grid_dependency_wait();
    const int items = *g.n_tasks * g.nmat * ipm;
    if (gt >= items) return;  // the whole team
    const int first_claim = static_cast<int>(gridDim.x) * kMvhWarps;

    // cursor over the stages to copy (it, p) and the item's expert / matrix / rows
    int cit = gt, cp = member;
    bool cfetch = false;
    uint32_t issued = 0, used = 0;
    int fifo_head = 0, fifo_tail = 0;
    auto issue = [&]() {
        const int task = cit / (g.nmat * ipm), rem = cit % (g.nmat * ipm);
        const int mi = rem / ipm, li = rem % ipm;
        const int e = g.tasks[task].expert;
        const int j = li & 7, G0 = (li >> 3) * kMvhRows;
        const int64_t off = (static_cast<int64_t>(j) * g.rowbytes + static_cast<int64_t>(cp) * SB) &
                            ~static_cast<int64_t>(15);
        const uint32_t slot = ring + (issued % kMvhNS) * kMvhSlot, bar = bars + 8 * (issued % kMvhNS);
        if (lane == 0) mbar_arrive_expect_tx(bar, NBX * BW * kMvhRows);
        __syncwarp();
        if (lane < NBX)
            tma_load_3d(slot + static_cast<uint32_t>(lane) * BW * kMvhRows, &g.map[mi],
                        static_cast<int>(off / 2) + static_cast<int>(BW / 2) * lane, G0, e, bar);
        ++issued;
        cp += ks;
        if (cp < stages) return;
        if (ks == 1) {
            cfetch = true;
        } else {
            cp = member;
            cit += nteams;
        }
    };
    for (int q = 0; q < kMvhNS - 1 && !cfetch && cit < items; ++q) issue();

    bool ok = true;
    int it = gt;
    while (it < items) {
        const int task = it / (g.nmat * ipm), rem = it % (g.nmat * ipm);
        const int mi = rem / ipm, li = rem % ipm;
        const MoeTask tk = g.tasks[task];
        const int j = li & 7, G0 = (li >> 3) * kMvhRows;
        const int bcols = g.split ? 2 * tk.n : tk.n;
        const int xrow = (g.split ? 2 * tk.pos : tk.pos) + gr % bcols;  // past the batch: a valid row
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int p = member; p < stages; p += ks) {
            if (cfetch) {
                int nx = 0;
                if (lane == 0) nx = first_claim + atomicAdd(g.ctr, 1);
                nx = __shfl_sync(0xffffffffu, nx, 0);
                cit = nx;
                cp = 0;
                cfetch = false;
                if (lane == 0) fifo[fifo_tail & 3] = nx;
                ++fifo_tail;
            }
            if (cit < items) {
                fence_proxy_async_smem();
                __syncwarp();
                issue();
            }
            const uint16_t* xr = g.xh + static_cast<int64_t>(xrow) * g.K + static_cast<int64_t>(p) * SK;
            const uint32_t slot = ring + (used % kMvhNS) * kMvhSlot;
            if (ok) ok = mvh_wait(bars + 8 * (used % kMvhNS), (used / kMvhNS) & 1u, g.st.err);
            ++used;
            const uint32_t L = static_cast<uint32_t>(
                (static_cast<int64_t>(j) * g.rowbytes + static_cast<int64_t>(p) * SB) & 15);
            if constexpr (FMT == FMT_Q6_K) q6k_stage(slot, gr, c, po, L, selc, xr, acc);
            else if constexpr (FMT == FMT_Q4_0) q4_0_stage(slot, gr, c, xr, acc);
            else q8_0_stage(slot, gr, c, L, xr, acc);
            __syncwarp();
        }
        if (ks > 1) {
#pragma unroll
            for (int q = 0; q < 4; ++q) part[(warp * 4 + q) * 32 + lane] = acc[q];
            mvh_team_sync(team, ks);
            if (member == 0) {
                for (int t2 = 1; t2 < ks; ++t2)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[q] += part[((warp + t2) * 4 + q) * 32 + lane];
            }
            mvh_team_sync(team, ks);
        }
        if (member == 0) {
            float* out = g.out[mi];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t n = static_cast<int64_t>(j) + 8 * (G0 + gr + 8 * h);
                if (n >= g.N) continue;
                if (g.split) {
                    // columns 2c, 2c + 1: token c's hi and lo rows
                    if (c < tk.n)
                        out[static_cast<int64_t>(tk.pos + c) * g.N + n] =
                            (acc[2 * h] + acc[2 * h + 1]) * g.xinv[tk.pos + c];
                } else {
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2) {
                        const int b = 2 * c + b2;
                        if (b < tk.n)
                            out[static_cast<int64_t>(tk.pos + b) * g.N + n] = acc[2 * h + b2] * g.xinv[tk.pos + b];
                    }
                }
            }
        }
        if (ks > 1) {
            it += nteams;
        } else {
            __syncwarp();
            it = fifo[fifo_head & 3];
            ++fifo_head;
        }
    }
    if (!ok)
        for (uint32_t u = used > kMvhNS ? used - kMvhNS : 0; u < issued; ++u)
            (void)mvh_wait(bars + 8 * (u % kMvhNS), (u / kMvhNS) & 1u, g.st.err);
}

// Largest magnitude of the block's values (fp32 bits of |v|, 0 if none),
// reduced over the CTA (blockDim.x a multiple of 32, at most 1024).
__device__ __forceinline__ float block_amax(float m) {
    __shared__ float red[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    return m;
}

// 2^s with the largest magnitude times 2^s in [2^14, 2^15) (1 for 0, inf, NaN)
__device__ __forceinline__ int fp16_exponent(float amax) {
    if (!(amax > 0.0f) || !(amax < INFINITY)) return 0;
    int e;
    (void)frexpf(amax, &e);
    return min(126, max(-126, 15 - e));
}

// gate/up prep: one CTA per grouped slot, the slot's token row (bf16) as
// scaled fp16 (8 values per 16-byte load); resets the matvec's item counter.
__global__ void __launch_bounds__(256) moe_prep_gu_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                          const int* __restrict__ pos_slot, int S,
                                                          uint16_t* __restrict__ xh, float* __restrict__ xinv,
                                                          int* ctr, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_GATHER);
    if (blockIdx.x == 0 && threadIdx.x == 0) *ctr = 0;
    for (int pos = blockIdx.x; pos < S; pos += gridDim.x) {
        const int slot = pos_slot[pos];
        if (slot < 0) continue;  // uniform over the CTA
        const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(slot / k) * H);
        uint4* out = reinterpret_cast<uint4*>(xh + static_cast<int64_t>(pos) * H);
        const int nv = H / 8;
        uint32_t mb = 0;  // magnitude bits of bf16 order like the magnitudes
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            const uint4 v = __ldg(xr + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) mb = max(mb, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
        }
        const int s = fp16_exponent(block_amax(__uint_as_float(mb << 16)));
        const float sc = ldexpf(1.0f, s);
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            const uint4 v = __ldg(xr + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __half lo = __float2half_rn(__uint_as_float(w[q] << 16) * sc);
                const __half hi = __float2half_rn(__uint_as_float(w[q] & 0xFFFF0000u) * sc);
                o[q] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
            }
            out[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (threadIdx.x == 0) xinv[pos] = ldexpf(1.0f, -s);
    }
}

// down prep: one CTA per grouped slot: h = silu(g) * u in fp32, as two fp16
// rows hi = fp16(h 2^s), lo = fp16(h 2^s - hi); resets the item counter. A
// thread keeps the h of its 4-value groups in registers between the two
// passes (I <= 256 * 4 * 8).
__global__ void __launch_bounds__(256) moe_prep_d_kernel(const float* __restrict__ gg, const float* __restrict__ uu,
                                                         int I, const int* __restrict__ pos_slot, int S,
                                                         uint16_t* __restrict__ xh, float* __restrict__ xinv,
                                                         int* ctr, DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_MOE_SILU);
    if (blockIdx.x == 0 && threadIdx.x == 0) *ctr = 0;
    constexpr int kPer = 8;  // 4-value groups per thread at most
    for (int pos = blockIdx.x; pos < S; pos += gridDim.x) {
        if (pos_slot[pos] < 0) continue;
        const float4* g4 = reinterpret_cast<const float4*>(gg + static_cast<int64_t>(pos) * I);
        const float4* u4 = reinterpret_cast<const float4*>(uu + static_cast<int64_t>(pos) * I);
        const int nv = I / 4;
        float4 h[kPer];
        float m = 0.0f;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = threadIdx.x + q * static_cast<int>(blockDim.x);
            h[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (i < nv) {
                const float4 gv = __ldg(g4 + i), uv = __ldg(u4 + i);
                h[q] = make_float4(gv.x / (1.0f + expf(-gv.x)) * uv.x, gv.y / (1.0f + expf(-gv.y)) * uv.y,
                                   gv.z / (1.0f + expf(-gv.z)) * uv.z, gv.w / (1.0f + expf(-gv.w)) * uv.w);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(h[q].x), fabsf(h[q].y)), fmaxf(fabsf(h[q].z), fabsf(h[q].w))));
            }
        }
        const int s = fp16_exponent(block_amax(m));
        const float sc = ldexpf(1.0f, s);
        uint2* hi_row = reinterpret_cast<uint2*>(xh + (2 * static_cast<int64_t>(pos)) * I);
        uint2* lo_row = reinterpret_cast<uint2*>(xh + (2 * static_cast<int64_t>(pos) + 1) * I);
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = threadIdx.x + q * static_cast<int>(blockDim.x);
            if (i >= nv) continue;
            const float v[4] = {h[q].x * sc, h[q].y * sc, h[q].z * sc, h[q].w * sc};
            uint32_t hb[4], lb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const __half hv = __float2half_rn(v[r]);
                hb[r] = __half_as_ushort(hv);
                lb[r] = __half_as_ushort(__float2half_rn(v[r] - __half2float(hv)));
            }
            hi_row[i] = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
            lo_row[i] = make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
        }
        if (threadIdx.x == 0) xinv[pos] = ldexpf(1.0f, -s);
    }
}

bool moe_mvh_supported(int fmt, int H, int I) {
    // (the down prep holds a slot's h in registers: I <= 256 threads x 8 x 4)
    return (fmt == FMT_Q4_0 || fmt == FMT_Q8_0 || fmt == FMT_Q6_K) && H % 256 == 0 && I % 256 == 0 &&
           I <= 256 * 8 * 4;
}

namespace {

struct MoeWs {
    uint16_t* xh_gu;
    float* xinv_gu;
    float* g;
    float* u;
    uint16_t* xh_d;
    float* xinv_d;
    int* ctr;
    size_t total;
};

MoeWs moe_ws_layout(uint8_t* base, int T, int k, int H, int I) {
    const size_t S = static_cast<size_t>(T) * k;
    MoeWs w{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + o : nullptr;
        o = round256(o + bytes);
        return p;
    };
    w.ctr = reinterpret_cast<int*>(take(4));
    w.xh_gu = reinterpret_cast<uint16_t*>(take(S * H * 2));
    w.xinv_gu = reinterpret_cast<float*>(take(S * 4));
    w.g = reinterpret_cast<float*>(take(S * I * 4));
    w.u = reinterpret_cast<float*>(take(S * I * 4));
    w.xh_d = reinterpret_cast<uint16_t*>(take(2 * S * I * 2));
    w.xinv_d = reinterpret_cast<float*>(take(S * 4));
    w.total = o;
    return w;
}

template <int FMT>
cudaError_t moe_mvh_prepare() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(moe_mvh_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kMvhSmem));
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(moe_mvh_kernel<FMT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
    });
    return err;
}

// a table as [E][N / 8][8 * rowbytes] 16-bit elements, boxes 16 rows high
cudaError_t moe_map(CUtensorMap* map, int fmt, const void* base, int64_t stride, int E, int64_t N,
                    int64_t rowbytes) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(4 * rowbytes), static_cast<cuuint64_t>(N / 8),
                                static_cast<cuuint64_t>(E)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(8 * rowbytes), static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[3] = {mvh_box_w(fmt) / 2, static_cast<cuuint32_t>(kMvhRows), 1u};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

template <int FMT>
cudaError_t moe_mvh_launch(MvhMoeArgs& a, int max_items, int sms, cudaStream_t s) {
    cudaError_t e = moe_mvh_prepare<FMT>();
    if (e != cudaSuccess) return e;
    // the K split depends on the shape only (never on the tokens), so a
    // token's output does not depend on which other tokens share the call
    const int stages = static_cast<int>(a.K / mvh_stage_k(FMT));
    a.ks = stages >= 16 ? 2 : 1;
    const int64_t per_cta = kMvhWarps / a.ks;
    const int grid = static_cast<int>(std::min<int64_t>(sms, (max_items + per_cta - 1) / per_cta));
    return launch_pdl(moe_mvh_kernel<FMT>, dim3(grid), dim3(kMvhWarps * 32), kMvhSmem, s, a);
}

}  // namespace

size_t moe_mvh_workspace_bytes(int T, int k, int H, int I) { return moe_ws_layout(nullptr, T, k, H, I).total; }

cudaError_t moe_mvh_run(int fmt, int E, int H, int I, int T, int k, const MvhMoeTables& tab, const void* x,
                        const int* n_tasks, const MoeTask* tasks, const int* pos_slot, void* ws, float* o,
                        int sms, cudaStream_t s, DevState st) {
    const int S = T * k;
    const MoeWs w = moe_ws_layout(static_cast<uint8_t*>(ws), T, k, H, I);
    const int64_t rb_gu = H / block_elems(fmt) * block_bytes(fmt), rb_d = I / block_elems(fmt) * block_bytes(fmt);
    // tasks at most: every slot its own task, or every expert one task per kMoeMvhTask tokens
    const int max_tasks = S;
    cudaError_t e = launch_pdl(moe_prep_gu_kernel, dim3(static_cast<unsigned>(S)), dim3(256), 0, s,
                               static_cast<const uint16_t*>(x), H, k, pos_slot, S, w.xh_gu, w.xinv_gu, w.ctr, st);
    if (e != cudaSuccess) return e;
    static thread_local MvhMoeArgs a;
    memset(&a, 0, sizeof a);
    a.n_tasks = n_tasks;
    a.tasks = tasks;
    a.ctr = w.ctr;
    a.st = st;
    // gate and up
    if ((e = moe_map(&a.map[0], fmt, tab.base[0], tab.stride[0], E, I, rb_gu)) != cudaSuccess) return e;
    if ((e = moe_map(&a.map[1], fmt, tab.base[1], tab.stride[1], E, I, rb_gu)) != cudaSuccess) return e;
    a.xh = w.xh_gu;
    a.xinv = w.xinv_gu;
    a.out[0] = w.g;
    a.out[1] = w.u;
    a.N = I;
    a.K = H;
    a.rowbytes = rb_gu;
    a.nmat = 2;
    a.split = 0;
    a.live_slot = QMM_LIVE_MOE_GATE_UP;
    int max_items = max_tasks * 2 * static_cast<int>((I + 8 * kMvhRows - 1) / (8 * kMvhRows) * 8);
    e = fmt == FMT_Q6_K ? moe_mvh_launch<FMT_Q6_K>(a, max_items, sms, s)
      : fmt == FMT_Q4_0 ? moe_mvh_launch<FMT_Q4_0>(a, max_items, sms, s)
                        : moe_mvh_launch<FMT_Q8_0>(a, max_items, sms, s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_prep_d_kernel, dim3(static_cast<unsigned>(S)), dim3(256), 0, s,
                   static_cast<const float*>(w.g), static_cast<const float*>(w.u), I, pos_slot, S, w.xh_d, w.xinv_d,
                   w.ctr, st);
    if (e != cudaSuccess) return e;
    // down
    if ((e = moe_map(&a.map[0], fmt, tab.base[2], tab.stride[2], E, H, rb_d)) != cudaSuccess) return e;
    a.xh = w.xh_d;
    a.xinv = w.xinv_d;
    a.out[0] = o;
    a.out[1] = nullptr;
    a.N = H;
    a.K = I;
    a.rowbytes = rb_d;
    a.nmat = 1;
    a.split = 1;
    a.live_slot = QMM_LIVE_MOE_DOWN;
    max_items = max_tasks * static_cast<int>((H + 8 * kMvhRows - 1) / (8 * kMvhRows) * 8);
    e = fmt == FMT_Q6_K ? moe_mvh_launch<FMT_Q6_K>(a, max_items, sms, s)
      : fmt == FMT_Q4_0 ? moe_mvh_launch<FMT_Q4_0>(a, max_items, sms, s)
                        : moe_mvh_launch<FMT_Q8_0>(a, max_items, sms, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmm
