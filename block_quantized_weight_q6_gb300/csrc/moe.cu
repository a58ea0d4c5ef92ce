// moe.cu -- routed-expert FFN over experts resident in device memory, and the
// top-k softmax router.
//
// "Chasing x100", section "Where the wall actually fell: inversion": the
// routed experts stay resident and are decoded in place, and per token only
// its top-k experts are touched. Here every selected expert's gate, up and
// down matrices are streamed from HBM once per call, however many of the
// tokens chose it:
//   1. plan:    the (token, slot) pairs are ordered by expert (counting sort,
//               ties kept in slot order) and cut into tasks of <= 2 tokens
//   2. gather:  activation rows copied into that expert-grouped order
//   3. gate_up: per (task, 4 rows of the intermediate dimension), the gate and
//               up rows are decoded side by side (the matvec kernel's decoders)
//               and h = silu(g) * u is formed in registers
//   4. down:    per (task, 4 rows of the hidden dimension), o = Wd h
//   5. combine: y[t] = sum_j gate[t][j] * o[t, j], summed in j order
#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "gemv_impl.cuh"

namespace qmm {

bool g_moe_mvh_enabled = true;

namespace {

// rows per item: a lane's activations serve every row of the item, so more
// rows mean fewer activation reads per weight byte; the two-slot rings of 12
// warps bound them (Q4_0 segments are 608 bytes, Q8_0 1120, q6_K 1712). The
// down projection (fp32 activations) gets the most; the fused gate/up kernel
// holds two matrices' rows per item.
template <int FMT, bool FUSED>
__host__ __device__ constexpr int moe_rows() {
    return FMT == FMT_Q6_K ? (FUSED ? 2 : 4) : FMT == FMT_Q8_0 ? (FUSED ? 4 : 8) : (FUSED ? 6 : 12);
}
constexpr int kMoeNB = 2;       // tokens per task
constexpr int kMoeSlots = 2;    // ring slots per warp

struct MoeTable {
    const uint8_t* p[3 * kMoeMaxExperts];  // gate[E], up[E], down[E]
};

struct MoeArgs {
    int E, H, I, T, k;
    int x_bf16;
    const int32_t* idx;   // [T][k]
    const float* gate;    // [T][k]
    const void* x;        // [T][H]
    float* y;             // [T][H]
    // workspace
    int task_nb;          // tokens per task at most
    int* n_tasks;         // [1]
    MoeTask* tasks;       // [T*k]
    int* slot_pos;        // [T*k] grouped position of slot (t, j)
    int* pos_slot;        // [T*k] slot of each grouped position (-1 past the used ones)
    void* xg;             // [T*k][H] grouped activations (x's type)
    float* h;             // [T*k][I]
    float* o;             // [T*k][H]
    DevState st;
};

}  // namespace

// ---------------------------------------------------------------- 1. plan
// One CTA. Slots s = t * k + j. rank(s) = earlier slots with the same expert;
// pos(s) = (slots of smaller experts) + rank(s).
__global__ void __launch_bounds__(1024) moe_plan_kernel(const MoeArgs a) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(a.st, QMM_LIVE_MOE_PLAN_SLOT);
    extern __shared__ int sm[];
    int* cnt = sm;                    // [E]
    int* off = cnt + a.E;             // [E] slot offsets
    int* toff = off + a.E;            // [E] task offsets
    int* eidx = toff + a.E;           // [S]
    const int S = a.T * a.k;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
    for (int s = threadIdx.x; s < a.T * a.k; s += blockDim.x) a.pos_slot[s] = -1;
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        int e = a.idx[s];
        if (e < 0 || e >= a.E) {
            atomicOr(a.st.err, DERR_MOE_BAD_INDEX);
            e = -1;
        }
        eidx[s] = e;
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive prefix sums over the experts of the slot counts (off) and of
    // the task counts (toff), a block-wide scan per chunk of blockDim.x
    // experts with the running totals carried between chunks
    __shared__ int wsum[2][32];
    __shared__ int carry[2];
    if (threadIdx.x == 0) carry[0] = carry[1] = 0;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    for (int e0 = 0; e0 < a.E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int c = e < a.E ? cnt[e] : 0;
        const int t = (c + a.task_nb - 1) / a.task_nb;
        int ic = c, it = t;  // inclusive scans within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vc = __shfl_up_sync(0xffffffffu, ic, o), vt = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                ic += vc;
                it += vt;
            }
        }
        __syncthreads();  // carry[] of the previous chunk is final, wsum[] is free
        if (lane == 31) {
            wsum[0][wid] = ic;
            wsum[1][wid] = it;
        }
        __syncthreads();
        if (wid == 0) {
            int sc = lane < nw ? wsum[0][lane] : 0, st = lane < nw ? wsum[1][lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int vc = __shfl_up_sync(0xffffffffu, sc, o), vt = __shfl_up_sync(0xffffffffu, st, o);
                if (lane >= o) {
                    sc += vc;
                    st += vt;
                }
            }
            if (lane < nw) {  // exclusive warp offsets
                wsum[0][lane] = sc - wsum[0][lane];
                wsum[1][lane] = st - wsum[1][lane];
            }
        }
        __syncthreads();
        if (e < a.E) {
            off[e] = carry[0] + wsum[0][wid] + ic - c;
            toff[e] = carry[1] + wsum[1][wid] + it - t;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {  // the chunk's totals
            carry[0] += wsum[0][wid] + ic;
            carry[1] += wsum[1][wid] + it;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) *a.n_tasks = carry[1];
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int e = eidx[s];
        if (e < 0) {
            a.slot_pos[s] = -1;
            continue;
        }
        int rank = 0;
        for (int q = 0; q < s; ++q) rank += (eidx[q] == e);
        const int pos = off[e] + rank;
        a.slot_pos[s] = pos;
        a.pos_slot[pos] = s;
        if (rank % a.task_nb == 0) {
            MoeTask t;
            t.expert = e;
            t.pos = pos;
            t.n = min(a.task_nb, cnt[e] - rank);
            a.tasks[toff[e] + rank / a.task_nb] = t;
        }
    }
}

// ---------------------------------------------------------------- 2. gather

__global__ void moe_gather_kernel(const MoeArgs a) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(a.st, QMM_LIVE_MOE_GATHER_SLOT);
    const int S = a.T * a.k;
    const int esz = a.x_bf16 ? 2 : 4;
    const int64_t words = static_cast<int64_t>(a.H) * esz / 16;  // 16-byte units per row
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < S * words;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i / words);
        const int64_t w = i % words;
        const int pos = a.slot_pos[s];
        if (pos < 0) continue;
        const int t = s / a.k;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.x) +
                                                          static_cast<int64_t>(t) * a.H * esz);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.xg) +
                                              static_cast<int64_t>(pos) * a.H * esz);
        dst[w] = src[w];
    }
}

// ---------------------------------------------------------------- 3/4. matvecs
// Work item = (task, group of moe_rows() rows). FUSED: the gate and up rows of
// the group are decoded together and the item stores h = silu(g) * u;
// otherwise the down rows, storing o.
template <int FMT, bool FUSED>
__global__ void __launch_bounds__(kGemvThreads) moe_mv_kernel(const MoeArgs a, const MoeTable tab) {
    using F = Fmt<FMT>;
    constexpr int R = moe_rows<FMT, FUSED>(), NB = kMoeNB, NS = kMoeSlots;
    constexpr int NM = FUSED ? 2 : 1;  // matrices per item
    constexpr int SEG = seg_stride<FMT>();
    constexpr int SLOT = SEG * R * NM;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem) + warp * (NS * SLOT);
    const uint32_t bars = smem_u32(smem) + kGemvWarps * NS * SLOT + warp * NS * 8;
    grid_launch_dependents();
    live_bump(a.st, FUSED ? QMM_LIVE_MOE_GATE_UP_SLOT : QMM_LIVE_MOE_DOWN_SLOT);
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // the plan (and, for down, h) comes from the previous kernels
    grid_dependency_wait();

    const int rows = FUSED ? a.I : a.H;     // output rows of each matrix
    const int Kd = FUSED ? a.H : a.I;       // reduction length
    const int64_t nb = Kd / F::BE;
    const int nchunks = static_cast<int>((nb + F::CB - 1) / F::CB);
    const int groups = (rows + R - 1) / R;
    const int64_t n_items = static_cast<int64_t>(*a.n_tasks) * groups;
    const int64_t mat_bytes = static_cast<int64_t>(rows) * nb * F::BB;
    const int64_t tb16 = mat_bytes & ~static_cast<int64_t>(15);
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kGemvWarps + warp;
    const int64_t tw = static_cast<int64_t>(gridDim.x) * kGemvWarps;

    // issue cursor (every lane tracks it; lane 0 copies)
    int64_t ic_item = gw;
    int ic_c = 0;
    uint32_t issued = 0;
    auto issue_next = [&]() {
        if (ic_item >= n_items) return;
        const uint32_t sidx = issued % NS;
        const uint32_t dst = ring + sidx * SLOT;
        const uint32_t bar = bars + 8 * sidx;
        const int task = static_cast<int>(ic_item / groups);
        const int64_t row0 = static_cast<int64_t>(ic_item % groups) * R;
        const int e = a.tasks[task].expert;
        const int64_t kb0 = static_cast<int64_t>(ic_c) * F::CB;
        const int64_t len = min(static_cast<int64_t>(F::CB), nb - kb0) * F::BB;
        // lane (mtx * R + r) copies row row0 + r of matrix mtx: from the
        // 16-byte boundary at or below its segment, with plain loads for the
        // bytes past the last 16-byte boundary of the matrix
        static_assert(NM * R <= 32, "one lane per row segment");
        const int mtx = lane / R, r = lane % R;
        const int64_t row = row0 + r;
        const bool mine = mtx < NM && row < rows;
        const uint8_t* W = !mine ? nullptr : (FUSED ? tab.p[mtx * a.E + e] : tab.p[2 * a.E + e]);
        int64_t s16 = 0, e16 = 0;
        uint32_t bytes = 0;
        if (mine) {
            const int64_t st = (row * nb + kb0) * F::BB;
            s16 = st & ~static_cast<int64_t>(15);
            e16 = min((st + len + 15) & ~static_cast<int64_t>(15), tb16);
            if (e16 > s16) bytes = static_cast<uint32_t>(e16 - s16);
            for (int64_t q = max(e16, s16); q < st + len; ++q)
                sts_u8(dst + (mtx * R + r) * SEG + static_cast<uint32_t>(q - s16), W[q]);
        }
        fence_proxy_async_smem();
        const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
        if (lane == 0) mbar_arrive_expect_tx(bar, total);
        __syncwarp();
        if (bytes) bulk_g2s(dst + (mtx * R + r) * SEG, W + s16, bytes, bar);
        ++issued;
        if (++ic_c >= nchunks) {
            ic_c = 0;
            ic_item += tw;
        }
    };
    for (int s = 0; s < NS; ++s) issue_next();

    uint32_t used = 0;
    for (int64_t item = gw; item < n_items; item += tw) {
        const MoeTask task = a.tasks[item / groups];
        const int64_t row0 = static_cast<int64_t>(item % groups) * R;
        // the activations of this task: n consecutive grouped rows
        GemvArgs ga{};
        ga.N = rows;
        ga.K = Kd;
        ga.nb = nb;
        ga.B = task.n;
        if (FUSED) {
            ga.x_bf16 = a.x_bf16;
            ga.x = static_cast<const uint8_t*>(a.xg) +
                   static_cast<int64_t>(task.pos) * a.H * (a.x_bf16 ? 2 : 4);
        } else {
            ga.x_bf16 = 0;
            ga.x = a.h + static_cast<int64_t>(task.pos) * a.I;
        }
        float acc[NM][R][NB];
#pragma unroll
        for (int mtx = 0; mtx < NM; ++mtx)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[mtx][r][b] = 0.0f;
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t sidx = used % NS;
            const int64_t kb0 = static_cast<int64_t>(c) * F::CB;
            const int ncb = static_cast<int>(min(static_cast<int64_t>(F::CB), nb - kb0));
            // Q4_0 / Q8_0: this chunk's activations are loaded once for all
            // the item's matrices, before the wait for its weights; the next
            // chunk's are pulled into L1 meanwhile
            float2 xv[NB][16];
            if constexpr (FMT != FMT_Q6_K) {
                chunk_x32<NB>(ga, kb0, ncb, lane, xv);
                if (c + 1 < nchunks) {
                    const int64_t kb1 = kb0 + F::CB;
                    chunk_x32_prefetch<NB>(ga, kb1, static_cast<int>(min(static_cast<int64_t>(F::CB), nb - kb1)),
                                           lane);
                }
            }
            if (!mbar_wait(bars + 8 * sidx, (used / NS) & 1u)) {
                for (uint32_t u = used + 1; u < issued; ++u)
                    (void)mbar_wait(bars + 8 * (u % NS), (u / NS) & 1u);
                if (lane == 0) atomicOr(a.st.err, DERR_MOE_TIMEOUT);
                return;
            }
#pragma unroll
            for (int mtx = 0; mtx < NM; ++mtx) {
                const uint32_t slot = ring + sidx * SLOT + mtx * R * SEG;
                if constexpr (FMT == FMT_Q6_K)
                    chunk_q6k_wide<false, NB, R>(ga, slot, row0, kb0, ncb, lane, acc[mtx]);
                else
                    chunk_q32_wide<FMT, NB, R>(ga, slot, row0, kb0, ncb, lane, xv, acc[mtx]);
            }
            __syncwarp();
            ++used;
            issue_next();
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float v0 = warp_sum(acc[0][r][b]);
                float v = v0;
                if (FUSED) {
                    const float u = warp_sum(acc[NM - 1][r][b]);
                    v = v0 / (1.0f + expf(-v0)) * u;  // silu(g) * u
                }
                if (lane == ((r * NB + b) & 31) && row < rows && b < task.n) {
                    if (FUSED)
                        a.h[static_cast<int64_t>(task.pos + b) * a.I + row] = v;
                    else
                        a.o[static_cast<int64_t>(task.pos + b) * a.H + row] = v;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- 5. combine

__global__ void moe_combine_kernel(const MoeArgs a) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(a.st, QMM_LIVE_MOE_COMBINE_SLOT);
    const int64_t total = static_cast<int64_t>(a.T) * a.H;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / a.H);
        const int64_t n = i % a.H;
        float acc = 0.0f;
        for (int j = 0; j < a.k; ++j) {
            const int pos = a.slot_pos[t * a.k + j];
            if (pos < 0) continue;
            acc = fmaf(a.gate[t * a.k + j], a.o[static_cast<int64_t>(pos) * a.H + n], acc);
        }
        a.y[i] = acc;
    }
}

// ---------------------------------------------------------------- router
// One warp per token: k rounds of a warp arg-max (ties to the lower expert
// index), then a softmax over the k selected logits in fp32.
__global__ void route_topk_softmax_kernel(const float* __restrict__ logits, int T, int E, int k,
                                          int32_t* __restrict__ idx, float* __restrict__ gate,
                                          DevState st) {
    grid_launch_dependents();
    grid_dependency_wait();
    live_bump(st, QMM_LIVE_ROUTE_SLOT);
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= T) return;
    const float* l = logits + static_cast<int64_t>(warp) * E;
    constexpr int kPer = kMoeMaxExperts / 32;
    unsigned taken = 0;  // bit i: expert lane + 32 i already chosen
    float sel_v[32];
    int sel_i[32];
    float lv[kPer];  // the lane's logits, read once
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        lv[i] = e < E ? l[e] : -INFINITY;
    }
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            if (e >= E || ((taken >> i) & 1u)) continue;
            const float v = lv[i];
            if (v > bv || (v == bv && e < bi)) {
                bv = v;
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_v[j] = bv;
        sel_i[j] = bi;
    }
    if (lane == 0) {
        const float mx = sel_v[0];
        float z = 0.0f;
        for (int j = 0; j < k; ++j) z += expf(sel_v[j] - mx);
        for (int j = 0; j < k; ++j) {
            idx[warp * k + j] = sel_i[j];
            gate[warp * k + j] = expf(sel_v[j] - mx) / z;
        }
    }
}

// ---------------------------------------------------------------- host side

// Workspace: the plan (task count, tasks, slot <-> position maps), the
// grouped slots' outputs o, then the intermediates of whichever expert path
// runs (the larger of the two is reserved).
size_t moe_workspace_bytes(int T, int k, int H, int I, bool x_bf16) {
    const size_t S = static_cast<size_t>(T) * k;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t plan = r256(sizeof(int)) + r256(S * sizeof(MoeTask)) + 2 * r256(S * sizeof(int)) + r256(S * H * 4);
    const size_t cuda_core = r256(S * H * (x_bf16 ? 2 : 4)) + r256(S * I * 4);
    const size_t mma = moe_mvh_workspace_bytes(T, k, H, I);
    return plan + (cuda_core > mma ? cuda_core : mma);
}

// The experts of a table lie at one fixed stride (a multiple of 16 bytes)?
static bool table_stride(const void* const* w, int E, int64_t bytes, int64_t* stride) {
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(w[0]);
    const int64_t st = E > 1 ? static_cast<int64_t>(reinterpret_cast<uintptr_t>(w[1]) - b0) : bytes;
    if (st < bytes || st % 16 != 0) return false;
    for (int e = 0; e < E; ++e)
        if (reinterpret_cast<uintptr_t>(w[e]) != b0 + static_cast<uintptr_t>(e) * static_cast<uintptr_t>(st))
            return false;
    *stride = st;
    return true;
}

static int mv_occupancy(void (*k)(const MoeArgs, const MoeTable), size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static std::map<std::pair<int, void (*)(const MoeArgs, const MoeTable)>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, k});
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kGemvThreads, smem) != cudaSuccess)
        n = 0;
    cache[{dev, k}] = n;
    return n;
}

template <int FMT>
static cudaError_t launch_mvs(const MoeArgs& a, const MoeTable& tab, int sms, cudaStream_t s) {
    constexpr int SEG = seg_stride<FMT>();
    for (int fused = 1; fused >= 0; --fused) {
        auto k = fused ? moe_mv_kernel<FMT, true> : moe_mv_kernel<FMT, false>;
        const int NM = fused ? 2 : 1;
        const int R = fused ? moe_rows<FMT, true>() : moe_rows<FMT, false>();
        const size_t smem = static_cast<size_t>(kGemvWarps) * kMoeSlots * SEG * R * NM +
                            kGemvWarps * kMoeSlots * 8;
        const int occ = mv_occupancy(k, smem);
        if (occ <= 0) return cudaErrorInvalidConfiguration;
        // enough warps for the largest possible task list (every slot its own task)
        const int rows = fused ? a.I : a.H;
        const int64_t max_items = static_cast<int64_t>(a.T) * a.k * ((rows + R - 1) / R);
        int64_t grid = (max_items + kGemvWarps - 1) / kGemvWarps;
        if (grid > static_cast<int64_t>(sms) * occ) grid = static_cast<int64_t>(sms) * occ;
        cudaError_t e = launch_pdl(k, dim3(static_cast<unsigned>(grid)), dim3(kGemvThreads), smem, s, a, tab);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t moe_launch(int fmt, int E, int H, int I, int T, int k, const void* const* wg,
                       const void* const* wu, const void* const* wd, const int32_t* idx,
                       const float* gate, const void* x, int x_bf16, float* y, void* ws, int sms,
                       cudaStream_t s, DevState st) {
    MoeArgs a{};
    a.E = E;
    a.H = H;
    a.I = I;
    a.T = T;
    a.k = k;
    a.x_bf16 = x_bf16;
    a.idx = idx;
    a.gate = gate;
    a.x = x;
    a.y = y;
    a.st = st;
    const size_t S = static_cast<size_t>(T) * k;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    uint8_t* p = static_cast<uint8_t*>(ws);
    a.n_tasks = reinterpret_cast<int*>(p);
    p += r256(sizeof(int));
    a.tasks = reinterpret_cast<MoeTask*>(p);
    p += r256(S * sizeof(MoeTask));
    a.slot_pos = reinterpret_cast<int*>(p);
    p += r256(S * sizeof(int));
    a.pos_slot = reinterpret_cast<int*>(p);
    p += r256(S * sizeof(int));
    a.o = reinterpret_cast<float*>(p);
    p += r256(S * H * 4);
    uint8_t* rest = p;
    a.xg = p;
    p += r256(S * H * (x_bf16 ? 2 : 4));
    a.h = reinterpret_cast<float*>(p);
    // the fp16-MMA expert matvecs: bf16 activations, expert tables at a fixed
    // stride, shapes the stages fit (otherwise the CUDA-core expert matvec)
    const int be = fmt == FMT_Q6_K ? 256 : 32, bb = fmt == FMT_Q6_K ? 210 : (fmt == FMT_Q4_0 ? 18 : 34);
    const int64_t gu_bytes = static_cast<int64_t>(I) * (H / be) * bb, d_bytes = static_cast<int64_t>(H) * (I / be) * bb;
    MvhMoeTables mt{};
    const bool mma = x_bf16 && moe_mvh_supported(fmt, H, I) && g_moe_mvh_enabled &&
                     table_stride(wg, E, gu_bytes, &mt.stride[0]) && table_stride(wu, E, gu_bytes, &mt.stride[1]) &&
                     table_stride(wd, E, d_bytes, &mt.stride[2]);
    a.task_nb = mma ? kMoeMvhTask : kMoeNB;
    MoeTable tab;
    for (int e = 0; e < E; ++e) {
        tab.p[e] = static_cast<const uint8_t*>(wg[e]);
        tab.p[E + e] = static_cast<const uint8_t*>(wu[e]);
        tab.p[2 * E + e] = static_cast<const uint8_t*>(wd[e]);
    }
    const size_t plan_smem = (3 * static_cast<size_t>(E) + S) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(moe_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan_smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_plan_kernel, dim3(1), dim3(1024), plan_smem, s, a);
    if (e != cudaSuccess) return e;
    if (mma) {
        mt.base[0] = wg[0];
        mt.base[1] = wu[0];
        mt.base[2] = wd[0];
        e = moe_mvh_run(fmt, E, H, I, T, k, mt, x, a.n_tasks, a.tasks, a.pos_slot, rest, a.o, sms, s, st);
        if (e != cudaSuccess) return e;
        int64_t cb = (static_cast<int64_t>(T) * H + 255) / 256;
        if (cb > 4 * sms) cb = 4 * sms;
        e = launch_pdl(moe_combine_kernel, dim3(static_cast<unsigned>(cb)), dim3(256), 0, s, a);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t gwords = static_cast<int64_t>(S) * H * (x_bf16 ? 2 : 4) / 16;
    int64_t gb = (gwords + 255) / 256;
    if (gb > 4 * sms) gb = 4 * sms;
    e = launch_pdl(moe_gather_kernel, dim3(static_cast<unsigned>(gb > 0 ? gb : 1)), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    e = fmt == FMT_Q6_K ? launch_mvs<FMT_Q6_K>(a, tab, sms, s)
                        : (fmt == FMT_Q4_0 ? launch_mvs<FMT_Q4_0>(a, tab, sms, s)
                                           : launch_mvs<FMT_Q8_0>(a, tab, sms, s));
    if (e != cudaSuccess) return e;
    int64_t cb = (static_cast<int64_t>(T) * H + 255) / 256;
    if (cb > 4 * sms) cb = 4 * sms;
    e = launch_pdl(moe_combine_kernel, dim3(static_cast<unsigned>(cb)), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t route_launch(const float* logits, int T, int E, int k, int32_t* idx, float* gate,
                         cudaStream_t s, DevState st) {
    const int threads = 128;
    const int blocks = (T * 32 + threads - 1) / threads;
    cudaError_t e = launch_pdl(route_topk_softmax_kernel, dim3(blocks), dim3(threads), 0, s, logits, T,
                               E, k, idx, gate, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmm
