// api.cu -- the C interface of libqmm (include/qmm.h): argument checks,
// launch planning, the W_exp plane registry and gate, liveness counters and
// error reporting. All compute runs in the kernels of the other files.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>
#include <algorithm>
#include <unordered_map>

#include "kernels.h"
#include "qmm.h"

using namespace qmm;

namespace qmm {
bool g_pdl_enabled = true;
}

// Library state that lives in device memory (one copy per device).
__device__ unsigned long long g_live[QMM_LIVE_COUNT];
__device__ unsigned int g_err;

// Scratch of qmm_gemv_noalloc: a fixed array in device memory (one copy per
// device that loads the library), so that entry point never allocates.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QMM_NOALLOC_SCRATCH_BYTES];

namespace {

thread_local cudaStream_t t_stream = nullptr;
thread_local void* t_ws = nullptr;
thread_local size_t t_ws_bytes = 0;
thread_local char t_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(QMM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- env gate
// Read once ("57 - r54 MINFER_MMQ_Q6K_EXP" section 3.1: the env is read
// exactly once, at load; unset means on, only an explicit "0" opts out).
struct Env {
    bool exp_on = true;
    bool debug_label = false;
    bool fault_plane_alloc = false;
    bool mv1_on = true;
    bool mv8_on = true;
    bool mvh_on = true;
    bool moe_grouped = true;  // one grouped GEMM launch per projection in moe_prefill
};
Env g_env;
std::once_flag g_env_once;

void read_env() {
    const char* e = std::getenv("QMM_Q6K_EXP");
    g_env.exp_on = !(e && std::strcmp(e, "0") == 0);
    const char* d = std::getenv("QMM_DEBUG_LABEL");
    g_env.debug_label = d && std::strcmp(d, "1") == 0;
    const char* f = std::getenv("QMM_FAULT");
    g_env.fault_plane_alloc = f && std::strcmp(f, "plane_alloc") == 0;
    const char* mv = std::getenv("QMM_MV1");
    g_env.mv1_on = !(mv && std::strcmp(mv, "0") == 0);
    const char* m8 = std::getenv("QMM_MV8");
    g_env.mv8_on = !(m8 && std::strcmp(m8, "0") == 0);
    const char* mm = std::getenv("QMM_MOE_MMA");
    qmm::g_moe_mvh_enabled = !(mm && std::strcmp(mm, "0") == 0);
    const char* mh = std::getenv("QMM_MVH");
    g_env.mvh_on = !(mh && std::strcmp(mh, "0") == 0);
    const char* mg = std::getenv("QMM_MOE_GROUPED");
    g_env.moe_grouped = !(mg && std::strcmp(mg, "0") == 0);
    const char* pdl = std::getenv("QMM_PDL");
    qmm::g_pdl_enabled = !(pdl && std::strcmp(pdl, "0") == 0);
}

// ---------------------------------------------------------------- devices
struct DevInfo {
    bool ready = false;
    int sms = 0;
    DevState st{};
};
constexpr int kMaxDev = 64;
DevInfo g_dev[kMaxDev];
std::mutex g_dev_mu;

int dev_info(DevInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDev) return fail(QMM_EUNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_live);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(live)");
        d.st.live = static_cast<unsigned long long*>(p);
        e = cudaGetSymbolAddress(&p, g_err);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(err)");
        d.st.err = static_cast<unsigned int*>(p);
        d.ready = true;
    }
    *out = &d;
    return QMM_OK;
}

// ---------------------------------------------------------------- plane registry
// Keyed by the weight pointer the GEMM receives (the key the page's engine
// had to get right, section 3.3), remembering the geometry the plane was
// built for so that a plane of another shape is never used silently.
struct PlaneEntry {
    const int8_t* plane;
    int64_t N, K;
};
std::unordered_map<const void*, PlaneEntry> g_planes;
std::mutex g_planes_mu;

// ---------------------------------------------------------------- formats
bool is_kquant(int f) { return f == FMT_Q4_K || f == FMT_Q2_K; }
int block_elems(int f) { return (f == FMT_Q6_K || is_kquant(f)) ? 256 : 32; }
int block_bytes(int f) {
    switch (f) {
        case FMT_Q6_K: return 210;
        case FMT_Q4_0: return 18;
        case FMT_Q4_K: return 144;
        case FMT_Q2_K: return 84;
        default: return 34;
    }
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int check_fmt(uint32_t fmt, int* wf, bool* bf16, bool* q8) {
    if (fmt & ~static_cast<uint32_t>(QMM_FMT_MASK | QMM_X_MASK | QMM_ACT_MASK))
        return fail(QMM_EINVAL, "fmt 0x%x has unknown bits", fmt);
    *wf = static_cast<int>(fmt & QMM_FMT_MASK);
    if (*wf != QMM_Q4_0 && *wf != QMM_Q8_0 && *wf != QMM_Q6_K && *wf != QMM_Q4_K && *wf != QMM_Q2_K)
        return fail(QMM_EINVAL, "unknown weight format 0x%x", fmt & QMM_FMT_MASK);
    const uint32_t xk = fmt & QMM_X_MASK, am = fmt & QMM_ACT_MASK;
    if (xk != QMM_X_F32 && xk != QMM_X_BF16)
        return fail(QMM_EINVAL, "unknown activation type 0x%x", xk);
    if (am != QMM_ACT_FLOAT && am != QMM_ACT_Q8)
        return fail(QMM_EINVAL, "unknown activation mode 0x%x", am);
    *bf16 = xk == QMM_X_BF16;
    *q8 = am == QMM_ACT_Q8;
    return QMM_OK;
}

// ---------------------------------------------------------------- matvec plan
// The tensor-core matvec (tcmv.cuh): work item = 128-row tile x a range of
// `sps` 256-wide K stages. The stage range is chosen so that the items fill
// the resident CTAs in whole waves, preferring long ranges (each item ends
// with one exposed accumulator drain); ranges shorter than K leave partial
// sums that a deterministic fixed-order reduction adds up.
struct GemvPlan {
    int NB, S, ncol, grid;
    int64_t nst, tiles, sps, pieces, items;
    size_t ws_xt, ws_xs, ws_part, ws_total;   // workspace byte offsets / total
};

int plan_gemv(int fmt, bool q8, bool bf16, int B, int64_t N, int64_t K, int sms, GemvPlan* p) {
    p->NB = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
    p->S = (q8 || bf16) ? 1 : 3;
    p->ncol = tcmv_ncol(p->NB, p->S);
    const int64_t nb = K / block_elems(fmt);
    const int bps = tcmv_stage_blocks(fmt);
    p->nst = (nb + bps - 1) / bps;
    p->tiles = (N + 127) / 128;
    const int occ = tcmv_occupancy(fmt, q8, p->NB, p->S);
    if (occ <= 0)
        return fail(QMM_ECUDA, "matvec kernel (fmt %d, NB %d, S %d) cannot launch", fmt, p->NB, p->S);
    const int64_t slots = static_cast<int64_t>(sms) * occ;
    double best = -1.0;
    int64_t best_sps = p->nst;
    for (int64_t sps = p->nst; sps >= 1; --sps) {
        const int64_t pieces = (p->nst + sps - 1) / sps;
        if (sps < p->nst && (pieces - 1) * sps >= p->nst) continue;  // same split as a longer sps
        const int64_t items = p->tiles * pieces;
        const int64_t waves = (items + slots - 1) / slots;
        const double fill = static_cast<double>(items) / static_cast<double>(waves * slots);
        const double score = fill * static_cast<double>(sps) / (static_cast<double>(sps) + 0.5);
        if (score > best + 1e-9) {
            best = score;
            best_sps = sps;
        }
    }
    p->sps = best_sps;
    p->pieces = (p->nst + p->sps - 1) / p->sps;
    p->items = p->tiles * p->pieces;
    p->grid = static_cast<int>(p->items < slots ? p->items : slots);
    size_t off = 0;
    // the prepared activation operand (q8 mode and fp32 float mode; bf16
    // float mode gathers its operand inside the matvec) and the q8 scales
    p->ws_xt = off;
    if (q8 || !bf16) off = round_up(off + static_cast<size_t>(p->nst) * p->ncol * 256 * 2, 256);
    p->ws_xs = off;
    if (q8) off = round_up(off + static_cast<size_t>(p->nst) * 8 * p->NB * 4, 256);
    p->ws_part = off;
    if (p->pieces > 1) off = round_up(off + static_cast<size_t>(p->pieces) * B * N * 4, 256);
    p->ws_total = off;
    return QMM_OK;
}

// Launches the activation layout (or quantizer), the matvec and, for partial
// sums, the reduction, with workspace `ws` (at least p.ws_total bytes).
int run_gemv(int wf, bool q8, bool bf16, const void* W, const void* x, float* y, int64_t N,
             int64_t K, int B, const GemvPlan& p, uint8_t* ws, const DevInfo* d) {
    TcmvArgs a{};
    a.W = static_cast<const uint8_t*>(W);
    a.N = N;
    a.K = K;
    a.nb = K / block_elems(wf);
    a.total_bytes = N * a.nb * block_bytes(wf);
    a.rowbytes = a.nb * block_bytes(wf);
    a.n8 = N / 8 * 8;
    a.x = x;
    a.x_bf16 = bf16 ? 1 : 0;
    const bool tile = q8 || !bf16;
    a.xt = tile ? reinterpret_cast<const uint16_t*>(ws + p.ws_xt) : nullptr;
    a.xs = q8 ? reinterpret_cast<const float*>(ws + p.ws_xs) : nullptr;
    a.B = B;
    a.y = y;
    a.part = p.pieces > 1 ? reinterpret_cast<float*>(ws + p.ws_part) : nullptr;
    a.tiles = p.tiles;
    a.nst = p.nst;
    a.sps = p.sps;
    a.pieces = p.pieces;
    a.items = p.items;
    a.st = d->st;
    a.live_slot = q8 ? QMM_LIVE_GEMV_Q8 : QMM_LIVE_GEMV_FLOAT;
    cudaError_t e;
    if (tile) {
        e = act_tile_launch(x, bf16, B, K, wf, p.NB, p.S, p.ncol, p.nst, q8,
                            const_cast<uint16_t*>(a.xt), const_cast<float*>(a.xs), t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "activation tile launch");
    }
    e = tcmv_launch(wf, q8, p.NB, p.S, p.grid, t_stream, a);
    if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
    if (p.pieces > 1) {
        e = splitk_reduce_launch(a.part, y, static_cast<int>(p.pieces), static_cast<int64_t>(B) * N,
                                 t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
    }
    return QMM_OK;
}

// ---------------------------------------------------------------- grouped matvec plan
// Several matvecs of one format and batch in one launch (tcmv over a
// TcmvGroup): one stage range `sps` for all of them, chosen by simulating
// the launch's round-robin walk of the items (CTA c takes items c, c + grid,
// ...): an item costs its stages plus kItemFill stage-times of pipeline fill
// and drain, and partial sums cost kReduce more for their reductions.
struct GroupPlan {
    int NB, S, ncol, grid, n;
    int64_t sps, items;
    int64_t nst[kTcMaxMats], tiles[kTcMaxMats], pieces[kTcMaxMats], item0[kTcMaxMats];
    size_t ws_xt[kTcMaxMats], ws_xs[kTcMaxMats], ws_part[kTcMaxMats], ws_total;
};

constexpr double kItemFill = 2.0, kReduce = 3.0;

double group_makespan(const GroupPlan& p, int64_t sps, int64_t slots, int64_t* items_out) {
    std::vector<double> cost;
    bool split = false;
    for (int m = 0; m < p.n; ++m) {
        const int64_t pieces = (p.nst[m] + sps - 1) / sps;
        split = split || pieces > 1;
        for (int64_t pc = 0; pc < pieces; ++pc) {
            const double c = static_cast<double>(std::min(sps, p.nst[m] - pc * sps)) + kItemFill;
            for (int64_t t = 0; t < p.tiles[m]; ++t) cost.push_back(c);
        }
    }
    const int64_t items = static_cast<int64_t>(cost.size());
    const int64_t grid = items < slots ? items : slots;
    double worst = 0.0;
    for (int64_t c = 0; c < grid; ++c) {
        double t = 0.0;
        for (int64_t i = c; i < items; i += grid) t += cost[i];
        worst = std::max(worst, t);
    }
    *items_out = items;
    return worst + (split ? kReduce : 0.0);
}

int plan_gemv_group(int fmt, bool q8, bool bf16, int B, int n, const int64_t* N, const int64_t* K, int sms,
                    GroupPlan* p) {
    p->n = n;
    p->NB = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
    p->S = (q8 || bf16) ? 1 : 3;
    p->ncol = tcmv_ncol(p->NB, p->S);
    const int bps = tcmv_stage_blocks(fmt);
    int64_t max_nst = 1;
    for (int m = 0; m < n; ++m) {
        p->nst[m] = (K[m] / block_elems(fmt) + bps - 1) / bps;
        p->tiles[m] = (N[m] + 127) / 128;
        max_nst = std::max(max_nst, p->nst[m]);
    }
    const int occ = tcmv_occupancy(fmt, q8, p->NB, p->S);
    if (occ <= 0)
        return fail(QMM_ECUDA, "matvec kernel (fmt %d, NB %d, S %d) cannot launch", fmt, p->NB, p->S);
    const int64_t slots = static_cast<int64_t>(sms) * occ;
    double best = 1e300;
    int64_t best_sps = max_nst, prev_pieces = -1;
    for (int64_t sps = max_nst; sps >= 1; --sps) {
        const int64_t pieces = (max_nst + sps - 1) / sps;
        if (pieces == prev_pieces) continue;  // the same split of the longest matrix
        prev_pieces = pieces;
        int64_t items = 0;
        const double t = group_makespan(*p, sps, slots, &items);
        if (t < best - 1e-9) {
            best = t;
            best_sps = sps;
        }
    }
    p->sps = best_sps;
    p->items = 0;
    size_t off = 0;
    for (int m = 0; m < n; ++m) {
        p->pieces[m] = (p->nst[m] + p->sps - 1) / p->sps;
        p->item0[m] = p->items;
        p->items += p->tiles[m] * p->pieces[m];
        p->ws_xt[m] = off;
        if (q8 || !bf16) off = round_up(off + static_cast<size_t>(p->nst[m]) * p->ncol * 256 * 2, 256);
        p->ws_xs[m] = off;
        if (q8) off = round_up(off + static_cast<size_t>(p->nst[m]) * 8 * p->NB * 4, 256);
        p->ws_part[m] = off;
        if (p->pieces[m] > 1) off = round_up(off + static_cast<size_t>(p->pieces[m]) * B * N[m] * 4, 256);
    }
    p->ws_total = off;
    p->grid = static_cast<int>(p->items < slots ? p->items : slots);
    return QMM_OK;
}

// Plans are cached per shape: the simulation costs a few hundred microseconds.
int plan_gemv_group_cached(int fmt, bool q8, bool bf16, int B, int n, const int64_t* N, const int64_t* K,
                           int sms, GroupPlan* p) {
    static std::mutex mu;
    static std::map<std::vector<int64_t>, GroupPlan> cache;
    std::vector<int64_t> key = {fmt, q8 ? 1 : 0, bf16 ? 1 : 0, B, n, sms};
    for (int m = 0; m < n; ++m) {
        key.push_back(N[m]);
        key.push_back(K[m]);
    }
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *p = it->second;
            return QMM_OK;
        }
    }
    int rc = plan_gemv_group(fmt, q8, bf16, B, n, N, K, sms, p);
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = *p;
    return QMM_OK;
}

int run_gemv_group(int wf, bool q8, bool bf16, const void* const* W, const void* const* x, float* const* y,
                   const int64_t* N, const int64_t* K, int B, const GroupPlan& p, uint8_t* ws,
                   const DevInfo* d) {
    static thread_local TcmvGroup g;  // large: kept off the stack
    g.nmat = p.n;
    g.items = p.items;
    g.st = d->st;
    g.live_slot = q8 ? QMM_LIVE_GEMV_Q8 : QMM_LIVE_GEMV_FLOAT;
    const bool tile = q8 || !bf16;
    ActTileSet ts{};
    ts.x_bf16 = bf16 ? 1 : 0;
    ts.B = B;
    ts.fmt = wf;
    ts.NB = p.NB;
    ts.S = p.S;
    ts.ncol = p.ncol;
    ts.q8 = q8 ? 1 : 0;
    cudaError_t e;
    for (int m = 0; m < p.n; ++m) {
        TcmvArgs& a = g.m[m];
        a = TcmvArgs{};
        a.W = static_cast<const uint8_t*>(W[m]);
        a.N = N[m];
        a.K = K[m];
        a.nb = K[m] / block_elems(wf);
        a.total_bytes = N[m] * a.nb * block_bytes(wf);
        a.rowbytes = a.nb * block_bytes(wf);
        a.n8 = N[m] / 8 * 8;
        a.x = x[m];
        a.x_bf16 = bf16 ? 1 : 0;
        a.xt = tile ? reinterpret_cast<const uint16_t*>(ws + p.ws_xt[m]) : nullptr;
        a.xs = q8 ? reinterpret_cast<const float*>(ws + p.ws_xs[m]) : nullptr;
        a.B = B;
        a.y = y[m];
        a.part = p.pieces[m] > 1 ? reinterpret_cast<float*>(ws + p.ws_part[m]) : nullptr;
        a.tiles = p.tiles[m];
        a.nst = p.nst[m];
        a.sps = p.sps;
        a.pieces = p.pieces[m];
        a.items = p.tiles[m] * p.pieces[m];
        a.item0 = p.item0[m];
        a.st = d->st;
        a.live_slot = g.live_slot;
        if (tile) {
            ts.x[ts.n] = x[m];
            ts.K[ts.n] = K[m];
            ts.xt[ts.n] = const_cast<uint16_t*>(a.xt);
            ts.xs[ts.n] = const_cast<float*>(a.xs);
            ts.start[ts.n] = ts.total;
            ts.total += p.nst[m] * 16 * p.ncol * 2;
            ++ts.n;
        }
    }
    if (ts.n > 0) {
        // every matrix's activation operand in one launch
        e = act_tile_set_launch(ts, t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "activation tile launch");
    }
    e = tcmv_launch_group(wf, q8, p.NB, p.S, p.grid, t_stream, g);
    if (e != cudaSuccess) return cuda_fail(e, "grouped matvec launch");
    // one reduction launch for all the split matrices of the group
    static_assert(kReduceSetMax >= kTcMaxMats, "a reduction set covers a group");
    SplitReduceSet rs{};
    for (int m = 0; m < p.n; ++m) {
        if (p.pieces[m] <= 1) continue;
        rs.part[rs.n] = g.m[m].part;
        rs.y[rs.n] = y[m];
        rs.count[rs.n] = static_cast<int64_t>(B) * N[m];
        rs.start[rs.n] = rs.total;
        rs.splits[rs.n] = static_cast<int>(p.pieces[m]);
        rs.total += rs.count[rs.n];
        ++rs.n;
    }
    if (rs.n > 0) {
        e = splitk_reduce_set_launch(rs, t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
    }
    return QMM_OK;
}

// ---------------------------------------------------------------- batch 1-8 matvecs
// Float mode, K % 256 == 0: bf16 activations, 1..8 rows and N % 8 == 0 go to
// the fp16-MMA matvec (mvh.cuh), every such matrix of a call in one launch
// whatever its format. The rest: one fp32 activation row to the CUDA-core
// matvec (mv1.cuh) when rows are whole 16-byte pieces (Q4_0, Q8_0; q6_K with
// K % 2048 == 0); 2..8 bf16 rows whose N is not a multiple of 8 to the
// bf16 warp-level MMA matvec (mv8.cuh); everything else to the
// tensor-memory matvec. QMM_MVH=0, QMM_MV1=0, QMM_MV8=0 switch a path off.
enum { FAST_NONE = 0, FAST_MV1 = 1, FAST_MV8 = 8, FAST_MVH = 16 };

int fast_path(int wf, bool q8, bool bf16, int B, int64_t N, int64_t K) {
    if (q8 || K % block_elems(wf) != 0) return FAST_NONE;
    if (bf16 && B <= 8 && g_env.mvh_on && mvh_supported(wf, N, K)) return FAST_MVH;
    const bool rows16 = (K / block_elems(wf) * block_bytes(wf)) % 16 == 0;
    if (B == 1 && rows16 && g_env.mv1_on && mv1_supported(wf, K)) return FAST_MV1;
    if (B >= 2 && B <= 8 && bf16 && g_env.mv8_on && mv8_supported(wf, K)) return FAST_MV8;
    return FAST_NONE;
}

// The K-quant ladder formats (Q4_K, Q2_K) run on the fp16-MMA matvec only.
bool kquant_runs(int wf, bool q8, bool bf16, int B, int64_t N, int64_t K) {
    return !is_kquant(wf) || fast_path(wf, q8, bf16, B, N, K) == FAST_MVH;
}

// Launches mv1 or mv8 over matrices sel[0 .. n-1] of the arrays.
int run_fast(int path, int wf, bool bf16, int B, int n, const int* sel, const void* const* W,
             const void* const* x, float* const* y, const int64_t* N, const int64_t* K, const DevInfo* d) {
    const int64_t rb = path == FAST_MV1 ? kMv1RowBlock : kMv8RowBlock;
    const int64_t piece = path == FAST_MV1 ? 2048 : 256;
    Mv1Group g{};
    g.nmat = n;
    g.x_bf16 = bf16 ? 1 : 0;
    g.B = B;
    g.st = d->st;
    g.live_slot = path == FAST_MV1 ? QMM_LIVE_GEMV_MV1 : QMM_LIVE_GEMV_MV8;
    int64_t items = 0;
    int min_pieces = 1 << 30;
    for (int i = 0; i < n; ++i) {
        const int m = sel[i];
        Mv1Mat& a = g.m[i];
        a.W = static_cast<const uint8_t*>(W[m]);
        a.x = x[m];
        a.y = y[m];
        a.N = N[m];
        a.K = K[m];
        a.rowbytes = K[m] / block_elems(wf) * block_bytes(wf);
        a.pieces = static_cast<int>((K[m] + piece - 1) / piece);
        a.full_pieces = static_cast<int>(K[m] / piece);
        a.aligned = a.rowbytes % 16 == 0 && reinterpret_cast<uintptr_t>(W[m]) % 16 == 0;
        a.item0 = static_cast<int>(items);
        items += (N[m] + rb - 1) / rb;
        min_pieces = std::min(min_pieces, a.pieces);
    }
    if (items > (int64_t{1} << 30)) return fail(QMM_EUNSUPPORTED, "matvec: %lld row blocks", (long long)items);
    g.items = static_cast<int>(items);
    const int occ = path == FAST_MV1 ? mv1_occupancy(wf) : mv8_occupancy(wf);
    if (occ <= 0) return fail(QMM_ECUDA, "matvec (fmt %d, path %d) cannot launch", wf, path);
    const int64_t slots = static_cast<int64_t>(d->sms) * occ;
    int grid = static_cast<int>(items < slots ? items : slots);
    g.ks = 1;
    if (path == FAST_MV8) {
        // warps per item: enough that the items keep every warp of the grid
        // busy, at most any matrix's stages
        const int64_t warps = slots * 8;
        while (g.ks < 8 && 2 * g.ks <= min_pieces && items * g.ks < warps) g.ks *= 2;
        const int64_t per_cta = 8 / g.ks;  // teams per CTA
        grid = static_cast<int>(std::min<int64_t>(slots, (items + per_cta - 1) / per_cta));
    }
    cudaError_t e = path == FAST_MV1 ? mv1_launch(wf, grid, t_stream, g) : mv8_launch(wf, grid, t_stream, g);
    if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
    return QMM_OK;
}

// Workspace of the fp16-MMA matvec for these matrices, as if no two shared
// their activations (the launch shares equal ones, so it never needs more).
size_t mvh_ws_bound(int n, const int* sel, const int64_t* K, int B) {
    size_t t = 256;  // the item counter
    for (int i = 0; i < n; ++i)
        t += round_up(static_cast<size_t>(B) * K[sel[i]] * 2, 256) + round_up(static_cast<size_t>(B) * 4, 256);
    return t;
}

// A set of matvecs of any formats wf[0 .. n-1] sharing activation type, mode
// and batch: the fp16-MMA matvec takes every matrix it can, in one launch;
// per format, the others go to the batch-1 / batch 2-8 kernels (one launch
// per K, so that each K gets the split its own items need) or to one
// tensor-memory matvec launch. Workspace regions follow each other in that
// order. With ws == nullptr nothing is launched and *need is set to the
// workspace the call needs.
int gemv_set(int n, const int* wf, bool q8, bool bf16, int B, const void* const* W, const void* const* x,
             float* const* y, const int64_t* N, const int64_t* K, const DevInfo* d, uint8_t* ws, size_t* need) {
    int path[kTcMaxMats];
    int hsel[kTcMaxMats], nh = 0;
    for (int m = 0; m < n; ++m) {
        path[m] = fast_path(wf[m], q8, bf16, B, N[m], K[m]);
        if (path[m] == FAST_MVH) hsel[nh++] = m;
    }
    size_t off = nh > 0 ? round_up(mvh_ws_bound(nh, hsel, K, B), 256) : 0;
    if (ws && nh > 0) {
        cudaError_t e = mvh_run(nh, hsel, wf, W, x, y, N, K, B, ws, d->sms, t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
    }
    for (int f : {QMM_Q4_0, QMM_Q8_0, QMM_Q6_K}) {
        // this format's matrices the batch-1 / batch 2-8 kernels take, one launch per K
        for (int i = 0; i < n; ++i) {
            if (wf[i] != f || (path[i] != FAST_MV1 && path[i] != FAST_MV8)) continue;
            bool first = true;
            for (int j = 0; j < i; ++j) first = first && !(wf[j] == f && path[j] == path[i] && K[j] == K[i]);
            if (!first) continue;
            int sel[kTcMaxMats], ns = 0;
            for (int j = i; j < n; ++j)
                if (wf[j] == f && path[j] == path[i] && K[j] == K[i]) sel[ns++] = j;
            if (ws) {
                int rc = run_fast(path[i], f, bf16, B, ns, sel, W, x, y, N, K, d);
                if (rc) return rc;
            }
        }
        // the rest of this format: one tensor-memory matvec launch
        const void* Wr[kTcMaxMats];
        const void* xr[kTcMaxMats];
        float* yr[kTcMaxMats];
        int64_t Nr[kTcMaxMats], Kr[kTcMaxMats];
        int nr = 0;
        for (int i = 0; i < n; ++i) {
            if (wf[i] != f || path[i] != FAST_NONE) continue;
            Wr[nr] = W ? W[i] : nullptr;
            xr[nr] = x ? x[i] : nullptr;
            yr[nr] = y ? y[i] : nullptr;
            Nr[nr] = N[i];
            Kr[nr] = K[i];
            ++nr;
        }
        if (nr == 0) continue;
        GroupPlan p;
        int rc = plan_gemv_group_cached(f, q8, bf16, B, nr, Nr, Kr, d->sms, &p);
        if (rc) return rc;
        if (ws) {
            rc = run_gemv_group(f, q8, bf16, Wr, xr, yr, Nr, Kr, B, p, ws + off, d);
            if (rc) return rc;
        }
        off = round_up(off + p.ws_total, 256);
    }
    *need = off;
    return QMM_OK;
}

// Checks the workspace a set needs against the one set, then runs it.
int gemv_set_run(const char* who, int n, const int* wf, bool q8, bool bf16, int B, const void* const* W,
                 const void* const* x, float* const* y, const int64_t* N, const int64_t* K, const DevInfo* d) {
    size_t need = 0;
    int rc = gemv_set(n, wf, q8, bf16, B, nullptr, nullptr, nullptr, N, K, d, nullptr, &need);
    if (rc) return rc;
    if (need > t_ws_bytes || (need && !t_ws))
        return fail(QMM_ENOWORKSPACE, "%s needs %zu bytes of workspace, %zu set", who, need, t_ws_bytes);
    return gemv_set(n, wf, q8, bf16, B, W, x, y, N, K, d, static_cast<uint8_t*>(t_ws), &need);
}

int check_gemv_args(uint32_t fmt, const void* W, const void* x, const float* y, int64_t N,
                    int64_t K, int B, int* wf, bool* bf16, bool* q8) {
    int rc = check_fmt(fmt, wf, bf16, q8);
    if (rc) return rc;
    if (!W || !x || !y) return fail(QMM_EINVAL, "null pointer (W %p, x %p, y %p)", W, x, (const void*)y);
    if (N <= 0 || K <= 0) return fail(QMM_EINVAL, "N %lld and K %lld must be positive",
                                      (long long)N, (long long)K);
    if (B < 1 || B > 16) return fail(QMM_EINVAL, "B = %d outside 1..16", B);
    if (K % block_elems(*wf)) return fail(QMM_EALIGN, "K = %lld is not a multiple of %d",
                                          (long long)K, block_elems(*wf));
    if (!aligned16(W) || !aligned16(x)) return fail(QMM_EALIGN, "W and x must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(y) & 3u) return fail(QMM_EALIGN, "y must be 4-byte aligned");
    if (!kquant_runs(*wf, *q8, *bf16, B, N, K))
        return fail(QMM_EUNSUPPORTED, "Q4_K / Q2_K matvecs need bf16 activations in float mode, B <= 8 "
                                      "and N %% 8 == 0 (the fp16-MMA matvec)");
    return QMM_OK;
}

// Arguments of a set of matvecs: formats may differ (multi) or not; the
// activation type and mode must agree.
int check_gemv_set(int n, const uint32_t* fmts, uint32_t fmt1, const void* const* W, const void* const* x,
                   float* const* y, const int64_t* N, const int64_t* K, int B, int* wf, bool* bf16, bool* q8) {
    if (n < 1 || n > kTcMaxMats) return fail(QMM_EINVAL, "n = %d outside 1..%d", n, kTcMaxMats);
    if (!W || !x || !y || !N || !K) return fail(QMM_EINVAL, "null array");
    for (int m = 0; m < n; ++m) {
        const uint32_t f = fmts ? fmts[m] : fmt1;
        if (fmts && m > 0 && (f & ~static_cast<uint32_t>(QMM_FMT_MASK)) !=
                                 (fmts[0] & ~static_cast<uint32_t>(QMM_FMT_MASK)))
            return fail(QMM_EINVAL, "matvec %d: activation type and mode differ from matvec 0", m);
        bool b16, aq8;
        int rc = check_gemv_args(f, W[m], x[m], y[m], N[m], K[m], B, &wf[m], &b16, &aq8);
        if (rc) return rc;
        *bf16 = b16;
        *q8 = aq8;
    }
    return QMM_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

int qmm_init(void) {
    std::call_once(g_env_once, read_env);
    return QMM_OK;
}

int qmm_set_stream(void* cuda_stream) {
    qmm_init();
    t_stream = static_cast<cudaStream_t>(cuda_stream);
    return QMM_OK;
}

int qmm_set_workspace(void* dev, size_t bytes) {
    qmm_init();
    if (!dev && bytes) return fail(QMM_EINVAL, "null workspace with %zu bytes", bytes);
    if (reinterpret_cast<uintptr_t>(dev) & 255u)
        return fail(QMM_EALIGN, "workspace must be 256-byte aligned");
    t_ws = dev;
    t_ws_bytes = dev ? bytes : 0;
    return QMM_OK;
}

size_t qmm_workspace_bytes(uint32_t fmt, int64_t M_or_B, int64_t N, int64_t K);

int qmm_gemv(uint32_t fmt, const void* W, const void* x, float* y, int64_t N, int64_t K, int B) {
    qmm_init();
    int wf;
    bool bf16, q8;
    int rc = check_gemv_args(fmt, W, x, y, N, K, B, &wf, &bf16, &q8);
    if (rc) return rc;
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    return gemv_set_run("qmm_gemv", 1, &wf, q8, bf16, B, &W, &x, &y, &N, &K, d);
}

int qmm_gemv_group(uint32_t fmt, int n, const void* const* W, const void* const* x, float* const* y,
                   const int64_t* N, const int64_t* K, int B) {
    qmm_init();
    int wf[kTcMaxMats];
    bool bf16 = false, q8 = false;
    int rc = check_gemv_set(n, nullptr, fmt, W, x, y, N, K, B, wf, &bf16, &q8);
    if (rc) return rc;
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    return gemv_set_run("qmm_gemv_group", n, wf, q8, bf16, B, W, x, y, N, K, d);
}

int qmm_gemv_multi(int n, const uint32_t* fmt, const void* const* W, const void* const* x, float* const* y,
                   const int64_t* N, const int64_t* K, int B) {
    qmm_init();
    int wf[kTcMaxMats];
    bool bf16 = false, q8 = false;
    if (!fmt) return fail(QMM_EINVAL, "null fmt array");
    int rc = check_gemv_set(n, fmt, 0, W, x, y, N, K, B, wf, &bf16, &q8);
    if (rc) return rc;
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    return gemv_set_run("qmm_gemv_multi", n, wf, q8, bf16, B, W, x, y, N, K, d);
}

static size_t set_workspace_bytes(int n, const uint32_t* fmts, uint32_t fmt1, const int64_t* N, const int64_t* K,
                                  int B) {
    qmm_init();
    if (n < 1 || n > kTcMaxMats || !N || !K || B < 1 || B > 16) return 0;
    int wf[kTcMaxMats];
    bool bf16 = false, q8 = false;
    for (int m = 0; m < n; ++m) {
        const uint32_t f = fmts ? fmts[m] : fmt1;
        if (check_fmt(f, &wf[m], &bf16, &q8)) return 0;
        if (N[m] <= 0 || K[m] <= 0 || K[m] % block_elems(wf[m])) return 0;
        if (!kquant_runs(wf[m], q8, bf16, B, N[m], K[m])) return 0;
    }
    DevInfo* d;
    if (dev_info(&d)) return 0;
    size_t need = 0;
    if (gemv_set(n, wf, q8, bf16, B, nullptr, nullptr, nullptr, N, K, d, nullptr, &need)) return 0;
    return need;
}

size_t qmm_gemv_group_workspace_bytes(uint32_t fmt, int n, const int64_t* N, const int64_t* K, int B) {
    return set_workspace_bytes(n, nullptr, fmt, N, K, B);
}

size_t qmm_gemv_multi_workspace_bytes(int n, const uint32_t* fmt, const int64_t* N, const int64_t* K, int B) {
    if (!fmt) return 0;
    return set_workspace_bytes(n, fmt, 0, N, K, B);
}

int qmm_quantize_q8(uint32_t x_type, const void* x, int64_t rows, int64_t K, int8_t* xq,
                    float* s) {
    qmm_init();
    if (x_type != QMM_X_F32 && x_type != QMM_X_BF16)
        return fail(QMM_EINVAL, "x_type 0x%x is not QMM_X_F32 or QMM_X_BF16", x_type);
    if (!x || !xq || !s) return fail(QMM_EINVAL, "null pointer");
    if (rows <= 0 || K <= 0) return fail(QMM_EINVAL, "rows and K must be positive");
    if (K % 32) return fail(QMM_EALIGN, "K = %lld is not a multiple of 32", (long long)K);
    if (!aligned16(x) || !aligned16(xq)) return fail(QMM_EALIGN, "x and xq must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(s) & 3u) return fail(QMM_EALIGN, "s must be 4-byte aligned");
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = quantize_q8_launch(x, x_type == QMM_X_BF16, rows, K, xq, s, nullptr, t_stream,
                                       d->st);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return QMM_OK;
}

size_t qmm_plane_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K);
}

int qmm_plane_wanted(int64_t N, int64_t K) {
    qmm_init();
    return (g_env.exp_on && N > 0 && K > 0 && K % 256 == 0) ? 1 : 0;
}

int qmm_plane_build(const void* W_q6k, int64_t N, int64_t K, int8_t* plane_dst) {
    qmm_init();
    if (!W_q6k) return fail(QMM_EINVAL, "null W");
    if (N <= 0 || K <= 0) return fail(QMM_EINVAL, "N and K must be positive");
    if (K % 256) return fail(QMM_EALIGN, "K = %lld is not a multiple of 256", (long long)K);
    if (!aligned16(W_q6k)) return fail(QMM_EALIGN, "W must be 16-byte aligned");
    if (plane_dst && !aligned16(plane_dst)) return fail(QMM_EALIGN, "plane must be 16-byte aligned");
    if (!plane_dst || g_env.fault_plane_alloc) {
        // a plane was wanted but none could be allocated: remember it so that
        // the in-kernel path taken later is labelled as a fallback
        std::lock_guard<std::mutex> lk(g_planes_mu);
        g_planes[W_q6k] = PlaneEntry{nullptr, N, K};
        std::fprintf(stderr, "qmm: W_exp plane for %p (%lld x %lld) not available; "
                             "q6_K GEMM falls back to in-kernel expansion\n",
                     W_q6k, (long long)N, (long long)K);
        return QMM_OK;
    }
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = plane_build_launch(static_cast<const uint8_t*>(W_q6k), N, K, plane_dst,
                                       t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "plane build launch");
    std::lock_guard<std::mutex> lk(g_planes_mu);
    g_planes[W_q6k] = PlaneEntry{plane_dst, N, K};
    return QMM_OK;
}

int qmm_plane_release(const void* W_q6k) {
    qmm_init();
    std::lock_guard<std::mutex> lk(g_planes_mu);
    g_planes.erase(W_q6k);
    return QMM_OK;
}

int qmm_gemm(uint32_t fmt, const void* W, const void* X, float* Y, int64_t M, int64_t N, int64_t K,
             const int8_t* exp_plane) {
    qmm_init();
    int wf;
    bool bf16, q8;
    int rc = check_fmt(fmt, &wf, &bf16, &q8);
    if (rc) return rc;
    if (wf != QMM_Q6_K && wf != QMM_Q4_0) return fail(QMM_EUNSUPPORTED, "qmm_gemm supports q6_K and Q4_0 weights");
    if (!W || !X || !Y) return fail(QMM_EINVAL, "null pointer (W %p, X %p, Y %p)", W, X, (void*)Y);
    if (M <= 0 || N <= 0 || K <= 0) return fail(QMM_EINVAL, "M, N, K must be positive");
    if (K % block_elems(wf))
        return fail(QMM_EALIGN, "K = %lld is not a multiple of %d", (long long)K, block_elems(wf));
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y))
        return fail(QMM_EALIGN, "W, X and Y must be 16-byte aligned");
    if (wf == QMM_Q4_0 && exp_plane) return fail(QMM_EINVAL, "Q4_0 has no W_exp plane");
    // which B path this launch takes ("57 - r54 MINFER_MMQ_Q6K_EXP" section 3.2 labels)
    int label = QMM_LIVE_GEMM_Q4_0;
    const char* label_name = "Q4_0 in-kernel-expand";
    if (wf == QMM_Q6_K) {
        std::lock_guard<std::mutex> lk(g_planes_mu);
        auto it = g_planes.find(W);
        if (exp_plane) {
            if (it == g_planes.end() || it->second.plane != exp_plane || it->second.N != N ||
                it->second.K != K)
                return fail(QMM_EPLANE, "exp_plane %p was not built for W %p (%lld x %lld)",
                            (const void*)exp_plane, W, (long long)N, (long long)K);
            label = QMM_LIVE_GEMM_EXP_PLANE;
            label_name = "W_exp-cp.async";
        } else if (it != g_planes.end()) {
            // a plane was wanted for this weight but is not here: failed
            // allocation, or a caller that lost it -- an accidental fallback
            label = QMM_LIVE_GEMM_FALLBACK;
            label_name = "in-kernel-expand(fallback!)";
        } else if (!g_env.exp_on) {
            label = QMM_LIVE_GEMM_EXP_OFF;
            label_name = "in-kernel-expand(exp=off)";
        } else {
            label = QMM_LIVE_GEMM_IN_KERNEL;
            label_name = "in-kernel-expand";
        }
    }
    if (g_env.debug_label)
        std::fprintf(stderr, "qmm: gemm %s M=%lld N=%lld K=%lld B path: %s\n",
                     wf == QMM_Q6_K ? "q6_K" : "Q4_0", (long long)M, (long long)N, (long long)K,
                     label_name);
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    const size_t a16b = round_up(gemm_a16_bytes(M, K), 256);
    const size_t xsb = round_up(static_cast<size_t>(M) * (K / 32) * 4, 256);
    const size_t need = a16b + xsb + round_up(gemm_part_bytes(M, N, K), 256);
    if (need > t_ws_bytes || !t_ws)
        return fail(QMM_ENOWORKSPACE, "qmm_gemm needs %zu bytes of workspace, %zu set", need,
                    t_ws_bytes);
    uint8_t* ws = static_cast<uint8_t*>(t_ws);
    uint16_t* a16 = reinterpret_cast<uint16_t*>(ws);
    float* xs = reinterpret_cast<float*>(ws + a16b);
    cudaError_t e = quantize_q8_launch(X, bf16, M, K, nullptr, xs, a16, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    float* part = gemm_part_bytes(M, N, K) ? reinterpret_cast<float*>(ws + a16b + xsb) : nullptr;
    e = gemm_launch(wf, exp_plane != nullptr, static_cast<const uint8_t*>(W), exp_plane, a16, xs, Y,
                    M, N, K, t_stream, d->st, label, part);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return QMM_OK;
}

int moe_gemv(uint32_t fmt, const qmm_moe_t* experts, const int32_t* idx, const float* gate_w,
             const void* x, float* y) {
    qmm_init();
    int wf;
    bool bf16, q8;
    int rc = check_fmt(fmt, &wf, &bf16, &q8);
    if (rc) return rc;
    if (q8) return fail(QMM_EUNSUPPORTED, "moe_gemv runs in float activation mode");
    if (is_kquant(wf)) return fail(QMM_EUNSUPPORTED, "moe_gemv supports q6_K, Q4_0 and Q8_0 experts");
    if (!experts || !experts->w_gate || !experts->w_up || !experts->w_down)
        return fail(QMM_EINVAL, "null expert table");
    const qmm_moe_t& m = *experts;
    if (m.n_experts < 1 || m.n_experts > kMoeMaxExperts)
        return fail(QMM_EINVAL, "n_experts = %d outside 1..%d", m.n_experts, kMoeMaxExperts);
    if (m.hidden <= 0 || m.inter <= 0 || m.n_tokens <= 0)
        return fail(QMM_EINVAL, "hidden, inter and n_tokens must be positive");
    if (m.top_k < 1 || m.top_k > 32 || m.top_k > m.n_experts)
        return fail(QMM_EINVAL, "top_k = %d outside 1..min(32, n_experts)", m.top_k);
    if (static_cast<int64_t>(m.n_tokens) * m.top_k > kMoeMaxSlots)
        return fail(QMM_EINVAL, "n_tokens * top_k = %lld exceeds %d per call",
                    static_cast<long long>(m.n_tokens) * m.top_k, kMoeMaxSlots);
    if (m.hidden % block_elems(wf) || m.inter % block_elems(wf))
        return fail(QMM_EALIGN, "hidden and inter must be multiples of %d", block_elems(wf));
    if (!idx || !gate_w || !x || !y) return fail(QMM_EINVAL, "null idx, gate_w, x or y");
    if (!aligned16(x)) return fail(QMM_EALIGN, "x must be 16-byte aligned");
    for (int e = 0; e < m.n_experts; ++e)
        if (!m.w_gate[e] || !m.w_up[e] || !m.w_down[e] || !aligned16(m.w_gate[e]) ||
            !aligned16(m.w_up[e]) || !aligned16(m.w_down[e]))
            return fail(QMM_EALIGN, "expert %d: matrices must be non-null and 16-byte aligned", e);
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    const size_t need = moe_workspace_bytes(m.n_tokens, m.top_k, m.hidden, m.inter, bf16);
    if (need > t_ws_bytes || !t_ws)
        return fail(QMM_ENOWORKSPACE, "moe_gemv needs %zu bytes of workspace, %zu set", need,
                    t_ws_bytes);
    cudaError_t e = moe_launch(wf, m.n_experts, m.hidden, m.inter, m.n_tokens, m.top_k, m.w_gate,
                               m.w_up, m.w_down, idx, gate_w, x, bf16, y, t_ws, d->sms, t_stream,
                               d->st);
    if (e != cudaSuccess) return cuda_fail(e, "moe launch");
    return QMM_OK;
}

}  // extern "C"

namespace {

constexpr int64_t kPrefillMaxSlots = int64_t{1} << 22;

// Workspace of moe_prefill, region by region (each rounded up to 256 B).
// The grouped flow pads every expert's rows to whole 128-row tiles, so its
// row regions hold up to S + 127 * min(E, S) rows.
struct PrefillWs {
    size_t counts, order, pos, xg, g, u, o, a16, xs, part, off, poff, tile, pos_pad, prow, total;
    int64_t rows;  // rows of the row regions
};

int64_t prefill_rows(int E, int64_t S, bool grouped) {
    return grouped ? (S + 127 * std::min<int64_t>(E, S) + 127) / 128 * 128 : S;
}

PrefillWs prefill_ws(int E, int64_t S, int H, int I, bool bf16, bool grouped) {
    PrefillWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    const int64_t Kmax = std::max(H, I);
    const int64_t R = prefill_rows(E, S, grouped);
    size_t part = 0;
    if (!grouped) {
        for (int64_t M = 128;; M += 128) {
            const int64_t m = std::min<int64_t>(M, S);
            part = std::max({part, gemm_part_bytes(m, I, H), gemm_part_bytes(m, H, I)});
            if (m == S) break;
        }
    }
    w.rows = R;
    w.counts = take(static_cast<size_t>(E) * 4);
    w.order = take(static_cast<size_t>(S) * 4);
    w.pos = take(static_cast<size_t>(S) * 4);
    w.xg = take(static_cast<size_t>(R) * H * (bf16 ? 2 : 4));
    w.g = take(static_cast<size_t>(R) * I * 4);
    w.u = take(static_cast<size_t>(R) * I * 4);
    w.o = take(static_cast<size_t>(R) * H * 4);
    w.a16 = take(gemm_a16_bytes(R, Kmax));
    w.xs = take(static_cast<size_t>(R) * (Kmax / 32) * 4);
    w.part = take(part);
    if (grouped) {
        w.off = take(static_cast<size_t>(E) * 4);
        w.poff = take(static_cast<size_t>(E) * 4);
        w.tile = take(static_cast<size_t>(R / 128) * 4);
        w.pos_pad = take(static_cast<size_t>(S) * 4);
        w.prow = take(static_cast<size_t>(R) * 4);
    }
    w.total = off;
    return w;
}

// Whether the table's matrices lie at one fixed stride (a multiple of 16
// bytes, at least a matrix apart): *stride is that stride.
bool table_stride(const void* const* w, int E, int64_t bytes, int64_t* stride) {
    if (E == 1) {
        *stride = static_cast<int64_t>(round_up(static_cast<size_t>(bytes), 16));
        return true;
    }
    const int64_t st = reinterpret_cast<intptr_t>(w[1]) - reinterpret_cast<intptr_t>(w[0]);
    if (st < bytes || st % 16) return false;
    for (int e = 2; e < E; ++e)
        if (reinterpret_cast<intptr_t>(w[e]) - reinterpret_cast<intptr_t>(w[e - 1]) != st) return false;
    *stride = st;
    return true;
}

// The grouped flow applies: the environment gate, and all three tables strided.
bool prefill_grouped(int wf, const qmm_moe_t& m, int64_t* sg, int64_t* su, int64_t* sd) {
    if (!g_env.moe_grouped) return false;
    const int64_t bg = static_cast<int64_t>(m.inter) * (m.hidden / block_elems(wf)) * block_bytes(wf);
    const int64_t bd = static_cast<int64_t>(m.hidden) * (m.inter / block_elems(wf)) * block_bytes(wf);
    return table_stride(m.w_gate, m.n_experts, bg, sg) && table_stride(m.w_up, m.n_experts, bg, su) &&
           table_stride(m.w_down, m.n_experts, bd, sd);
}

int check_prefill(uint32_t fmt, const qmm_moe_t* experts, int* wf, bool* bf16) {
    bool q8;
    int rc = check_fmt(fmt, wf, bf16, &q8);
    if (rc) return rc;
    if (*wf != QMM_Q4_0 && *wf != QMM_Q6_K)
        return fail(QMM_EUNSUPPORTED, "moe_prefill supports q6_K and Q4_0 experts (the prefill GEMM's formats)");
    if (!experts || !experts->w_gate || !experts->w_up || !experts->w_down)
        return fail(QMM_EINVAL, "null expert table");
    const qmm_moe_t& m = *experts;
    if (m.n_experts < 1 || m.n_experts > kMoeMaxExperts)
        return fail(QMM_EINVAL, "n_experts = %d outside 1..%d", m.n_experts, kMoeMaxExperts);
    if (m.hidden <= 0 || m.inter <= 0 || m.n_tokens <= 0)
        return fail(QMM_EINVAL, "hidden, inter and n_tokens must be positive");
    if (m.top_k < 1 || m.top_k > 32 || m.top_k > m.n_experts)
        return fail(QMM_EINVAL, "top_k = %d outside 1..min(32, n_experts)", m.top_k);
    if (static_cast<int64_t>(m.n_tokens) * m.top_k > kPrefillMaxSlots)
        return fail(QMM_EINVAL, "n_tokens * top_k = %lld exceeds %lld per call",
                    static_cast<long long>(m.n_tokens) * m.top_k, static_cast<long long>(kPrefillMaxSlots));
    const int be = std::max(block_elems(*wf), 32);
    if (m.hidden % be || m.inter % be) return fail(QMM_EALIGN, "hidden and inter must be multiples of %d", be);
    for (int e = 0; e < m.n_experts; ++e)
        if (!aligned16(m.w_gate[e]) || !aligned16(m.w_up[e]) || !aligned16(m.w_down[e]) || !m.w_gate[e] ||
            !m.w_up[e] || !m.w_down[e])
            return fail(QMM_EALIGN, "expert %d: weights must be non-null and 16-byte aligned", e);
    return QMM_OK;
}

}  // namespace

extern "C" {

size_t qmm_moe_prefill_workspace_bytes(uint32_t fmt, const qmm_moe_t* experts) {
    qmm_init();
    int wf;
    bool bf16;
    if (check_prefill(fmt, experts, &wf, &bf16)) return 0;
    const qmm_moe_t& m = *experts;
    int64_t sg, su, sd;
    const bool grouped = prefill_grouped(wf, m, &sg, &su, &sd);
    return prefill_ws(m.n_experts, static_cast<int64_t>(m.n_tokens) * m.top_k, m.hidden, m.inter, bf16, grouped)
        .total;
}

int moe_prefill(uint32_t fmt, const qmm_moe_t* experts, const int32_t* idx, const float* gate_w, const void* x,
                float* y) {
    qmm_init();
    int wf;
    bool bf16;
    int rc = check_prefill(fmt, experts, &wf, &bf16);
    if (rc) return rc;
    if (!idx || !gate_w || !x || !y) return fail(QMM_EINVAL, "null idx, gate_w, x or y");
    if (!aligned16(x) || !aligned16(y)) return fail(QMM_EALIGN, "x and y must be 16-byte aligned");
    const qmm_moe_t& m = *experts;
    const int E = m.n_experts, H = m.hidden, I = m.inter, T = m.n_tokens, k = m.top_k;
    const int64_t S = static_cast<int64_t>(T) * k;
    int64_t sg = 0, su = 0, sd = 0;
    const bool grouped = prefill_grouped(wf, m, &sg, &su, &sd);
    const PrefillWs w = prefill_ws(E, S, H, I, bf16, grouped);
    if (w.total > t_ws_bytes || !t_ws)
        return fail(QMM_ENOWORKSPACE, "moe_prefill needs %zu bytes of workspace, %zu set", w.total, t_ws_bytes);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(t_stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return fail(QMM_EUNSUPPORTED, "moe_prefill reads the expert counts on the host: it cannot be captured");
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    uint8_t* ws = static_cast<uint8_t*>(t_ws);
    int* counts = reinterpret_cast<int*>(ws + w.counts);
    int* order = reinterpret_cast<int*>(ws + w.order);
    int* pos = reinterpret_cast<int*>(ws + w.pos);
    uint8_t* Xg = ws + w.xg;
    float* G = reinterpret_cast<float*>(ws + w.g);
    float* U = reinterpret_cast<float*>(ws + w.u);
    float* O = reinterpret_cast<float*>(ws + w.o);
    uint16_t* a16 = reinterpret_cast<uint16_t*>(ws + w.a16);
    float* xs = reinterpret_cast<float*>(ws + w.xs);
    float* part = reinterpret_cast<float*>(ws + w.part);
    const int label = wf == QMM_Q4_0 ? QMM_LIVE_GEMM_Q4_0 : (g_env.exp_on ? QMM_LIVE_GEMM_IN_KERNEL : QMM_LIVE_GEMM_EXP_OFF);

    // the slots by expert, and each expert's count on the host
    cudaError_t e = moe_prefill_plan_launch(idx, static_cast<int>(S), E, counts, order, pos, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_prefill plan launch");
    std::vector<int> cnt(static_cast<size_t>(E));
    e = cudaMemcpyAsync(cnt.data(), counts, static_cast<size_t>(E) * 4, cudaMemcpyDeviceToHost, t_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(t_stream);
    if (e != cudaSuccess) return cuda_fail(e, "moe_prefill counts");
    int64_t total = 0;
    for (int c : cnt) total += c;
    if (total != S) return fail(QMM_EINVAL, "moe_prefill: %lld of %lld routing slots name an expert outside 0..%d",
                                static_cast<long long>(S - total), static_cast<long long>(S), E - 1);

    const int64_t xrow = static_cast<int64_t>(H) * (bf16 ? 2 : 4);
    if (grouped) {
        // every expert's rows padded to whole 128-row tiles: one GEMM launch
        // per projection over all experts, the weights of tile mt those of
        // expert tile[mt] (a tensor map over the strided table)
        static thread_local std::vector<int> hoff, hpoff, htile;
        hoff.assign(static_cast<size_t>(E), 0);
        hpoff.assign(static_cast<size_t>(E), 0);
        htile.clear();
        int64_t o = 0, po = 0;
        for (int ex = 0; ex < E; ++ex) {
            hoff[static_cast<size_t>(ex)] = static_cast<int>(o);
            hpoff[static_cast<size_t>(ex)] = static_cast<int>(po);
            const int64_t n = cnt[static_cast<size_t>(ex)];
            for (int64_t t = 0; t < (n + 127) / 128; ++t) htile.push_back(ex);
            o += n;
            po += (n + 127) / 128 * 128;
        }
        const int64_t R = po;  // padded rows
        int* doff = reinterpret_cast<int*>(ws + w.off);
        int* dpoff = reinterpret_cast<int*>(ws + w.poff);
        int* dtile = reinterpret_cast<int*>(ws + w.tile);
        int* pos_pad = reinterpret_cast<int*>(ws + w.pos_pad);
        int* prow = reinterpret_cast<int*>(ws + w.prow);
        e = cudaMemcpyAsync(doff, hoff.data(), static_cast<size_t>(E) * 4, cudaMemcpyHostToDevice, t_stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dpoff, hpoff.data(), static_cast<size_t>(E) * 4, cudaMemcpyHostToDevice, t_stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dtile, htile.data(), htile.size() * 4, cudaMemcpyHostToDevice, t_stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(prow, 0xFF, static_cast<size_t>(R) * 4, t_stream);
        if (e == cudaSuccess)
            e = moe_prefill_padmap_launch(idx, pos, doff, dpoff, static_cast<int>(S), pos_pad, prow, d->sms, t_stream,
                                          d->st);
        if (e == cudaSuccess)
            e = moe_prefill_gather_pad_launch(x, xrow, prow, k, static_cast<int>(R), Xg, d->sms, t_stream, d->st);
        if (e == cudaSuccess) e = quantize_q8_launch(Xg, bf16 ? 1 : 0, R, H, nullptr, xs, a16, t_stream, d->st);
        const uint8_t* g0 = static_cast<const uint8_t*>(m.w_gate[0]);
        const uint8_t* u0 = static_cast<const uint8_t*>(m.w_up[0]);
        const uint8_t* d0 = static_cast<const uint8_t*>(m.w_down[0]);
        if (e == cudaSuccess)
            e = gemm_grouped_launch(wf, g0, sg, E, dtile, a16, xs, G, R, I, H, t_stream, d->st, label);
        if (e == cudaSuccess)
            e = gemm_grouped_launch(wf, u0, su, E, dtile, a16, xs, U, R, I, H, t_stream, d->st, label);
        if (e == cudaSuccess) e = moe_prefill_silu_launch(G, U, R * I, d->sms, t_stream, d->st);
        if (e == cudaSuccess) e = quantize_q8_launch(G, 0, R, I, nullptr, xs, a16, t_stream, d->st);
        if (e == cudaSuccess)
            e = gemm_grouped_launch(wf, d0, sd, E, dtile, a16, xs, O, R, H, I, t_stream, d->st, label);
        if (e == cudaSuccess) e = moe_prefill_combine_launch(O, pos_pad, gate_w, T, k, H, y, t_stream, d->st);
        if (e != cudaSuccess) return cuda_fail(e, "moe_prefill grouped launch");
        return QMM_OK;
    }
    // gate and up: each expert's rows through the prefill GEMM
    e = moe_prefill_gather_launch(x, xrow, order, k, static_cast<int>(S), Xg, d->sms, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_prefill gather launch");
    auto gemm = [&](const void* W, const void* X, bool xb16, float* Y, int64_t M, int64_t N, int64_t K) {
        cudaError_t r = quantize_q8_launch(X, xb16 ? 1 : 0, M, K, nullptr, xs, a16, t_stream, d->st);
        if (r == cudaSuccess)
            r = gemm_launch(wf, false, static_cast<const uint8_t*>(W), nullptr, a16, xs, Y, M, N, K, t_stream, d->st,
                            label, gemm_part_bytes(M, N, K) ? part : nullptr);
        return r;
    };
    int64_t off = 0;
    for (int ex = 0; ex < E; ++ex) {
        const int64_t n = cnt[static_cast<size_t>(ex)];
        if (n == 0) continue;
        const uint8_t* Xe = Xg + off * xrow;
        e = gemm(m.w_gate[ex], Xe, bf16, G + off * I, n, I, H);
        if (e == cudaSuccess)
            e = gemm_launch(wf, false, static_cast<const uint8_t*>(m.w_up[ex]), nullptr, a16, xs, U + off * I, n, I,
                            H, t_stream, d->st, label, gemm_part_bytes(n, I, H) ? part : nullptr);
        if (e != cudaSuccess) return cuda_fail(e, "moe_prefill gate/up launch");
        off += n;
    }
    // h = silu(g) * u, then down: each expert's h rows through the GEMM
    e = moe_prefill_silu_launch(G, U, S * I, d->sms, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_prefill silu launch");
    off = 0;
    for (int ex = 0; ex < E; ++ex) {
        const int64_t n = cnt[static_cast<size_t>(ex)];
        if (n == 0) continue;
        e = gemm(m.w_down[ex], G + off * I, false, O + off * H, n, H, I);
        if (e != cudaSuccess) return cuda_fail(e, "moe_prefill down launch");
        off += n;
    }
    e = moe_prefill_combine_launch(O, pos, gate_w, T, k, H, y, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_prefill combine launch");
    return QMM_OK;
}

}  // extern "C"

namespace {

int check_cbk(int M, int64_t N, int64_t K, int B) {
    if (M != 2 && M != 3) return fail(QMM_EINVAL, "n_books = %d: 2 or 3 codebooks", M);
    if (N <= 0 || K <= 0) return fail(QMM_EINVAL, "N %lld and K %lld must be positive", (long long)N, (long long)K);
    if (B < 1 || B > 8) return fail(QMM_EINVAL, "B = %d outside 1..8", B);
    if (K % 128) return fail(QMM_EALIGN, "K = %lld is not a multiple of 128", (long long)K);
    if (N > (int64_t{1} << 31) / 8) return fail(QMM_EINVAL, "N = %lld too large", (long long)N);
    return QMM_OK;
}

}  // namespace

extern "C" {

size_t qmm_cbk_workspace_bytes(int n_books, int64_t N, int64_t K, int B) {
    qmm_init();
    if (check_cbk(n_books, N, K, B)) return 0;
    return round_up(cbk_part_bytes(n_books, N, K, B), 256);
}

int qmm_cbk_gemv(int n_books, const uint8_t* codes, const uint16_t* books, const uint16_t* scales, uint32_t x_type,
                 const void* x, float* y, int64_t N, int64_t K, int B) {
    qmm_init();
    int rc = check_cbk(n_books, N, K, B);
    if (rc) return rc;
    if (x_type != QMM_X_F32 && x_type != QMM_X_BF16) return fail(QMM_EINVAL, "x_type 0x%x", x_type);
    if (!codes || !books || !scales || !x || !y) return fail(QMM_EINVAL, "null pointer");
    if (!aligned16(codes) || !aligned16(books) || !aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 3u) ||
        (reinterpret_cast<uintptr_t>(scales) & 1u))
        return fail(QMM_EALIGN, "codes, books and x must be 16-byte aligned, y 4-byte, scales 2-byte");
    const size_t need = round_up(cbk_part_bytes(n_books, N, K, B), 256);
    if (need > t_ws_bytes || !t_ws)
        return fail(QMM_ENOWORKSPACE, "qmm_cbk_gemv needs %zu bytes of workspace, %zu set", need, t_ws_bytes);
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    cudaError_t e = cbk_launch(n_books, codes, books, scales, x, x_type == QMM_X_BF16 ? 1 : 0, y, N, K, B,
                               static_cast<float*>(t_ws), d->sms, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "cbk launch");
    return QMM_OK;
}

size_t qmm_moe_workspace_bytes(const qmm_moe_t* experts) {
    if (!experts || experts->n_tokens <= 0 || experts->top_k <= 0 || experts->hidden <= 0 ||
        experts->inter <= 0)
        return 0;
    return moe_workspace_bytes(experts->n_tokens, experts->top_k, experts->hidden, experts->inter,
                               false);
}

int qmm_route_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx, float* gate_w) {
    qmm_init();
    if (!logits || !idx || !gate_w) return fail(QMM_EINVAL, "null pointer");
    if (T < 1 || E < 1 || E > kMoeMaxExperts)
        return fail(QMM_EINVAL, "T = %d, E = %d (1 <= E <= %d)", T, E, kMoeMaxExperts);
    if (k < 1 || k > 32 || k > E) return fail(QMM_EINVAL, "k = %d outside 1..min(32, E)", k);
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = route_launch(logits, T, E, k, idx, gate_w, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    return QMM_OK;
}

size_t qmm_workspace_bytes(uint32_t fmt, int64_t M_or_B, int64_t N, int64_t K) {
    qmm_init();
    int wf;
    bool bf16, q8;
    if (check_fmt(fmt, &wf, &bf16, &q8)) return 0;
    if (M_or_B < 1 || N <= 0 || K <= 0 || K % block_elems(wf)) return 0;
    if (is_kquant(wf)) {
        if (M_or_B > 8 || !kquant_runs(wf, q8, bf16, static_cast<int>(M_or_B), N, K)) return 0;
    }
    // the GEMM's quantized activations (fp16 tiles + scales)
    size_t gemm = 0;
    if (wf == QMM_Q6_K || wf == QMM_Q4_0)
        gemm = round_up(gemm_a16_bytes(M_or_B, K), 256) +
               round_up(static_cast<size_t>(M_or_B) * (K / 32) * 4, 256) +
               round_up(gemm_part_bytes(M_or_B, N, K), 256);
    if (M_or_B > 16) return gemm;
    DevInfo* d;
    if (dev_info(&d)) return gemm;
    size_t need = 0;
    if (gemv_set(1, &wf, q8, bf16, static_cast<int>(M_or_B), nullptr, nullptr, nullptr, &N, &K, d, nullptr,
                 &need))
        return gemm;
    return need > gemm ? need : gemm;
}

int qmm_liveness_read(int64_t* counts, int n) {
    qmm_init();
    if (!counts || n < 0 || n > QMM_LIVE_COUNT)
        return fail(QMM_EINVAL, "counts must hold n <= %d values", QMM_LIVE_COUNT);
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    unsigned long long tmp[QMM_LIVE_COUNT];
    cudaError_t e = cudaMemcpy(tmp, d->st.live, sizeof tmp, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "liveness read");
    for (int i = 0; i < n; ++i) counts[i] = static_cast<int64_t>(tmp[i]);
    return QMM_OK;
}

int qmm_liveness_reset(void) {
    qmm_init();
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = cudaMemsetAsync(d->st.live, 0, sizeof(unsigned long long) * QMM_LIVE_COUNT,
                                    t_stream);
    if (e != cudaSuccess) return cuda_fail(e, "liveness reset");
    return QMM_OK;
}

int qmm_sync_check(void) {
    qmm_init();
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(t_stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned int err = 0;
    e = cudaMemcpy(&err, d->st.err, sizeof err, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "error word read");
    if (err) {
        unsigned int zero = 0;
        cudaMemcpy(d->st.err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (err & DERR_MOE_BAD_INDEX)
            return fail(QMM_EINVAL, "moe_gemv / moe_prefill: an expert index was outside 0..n_experts-1; "
                                    "its slot contributed nothing (flags 0x%x)", err);
        return fail(QMM_EDEVICE_TIMEOUT, "a kernel gave up a bounded wait (flags 0x%x)", err);
    }
    return QMM_OK;
}

// The device address of g_noalloc_scratch on the current device, looked up
// once per device (host code cannot use the symbol itself as an address).
static int noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDev) return fail(QMM_EUNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
        addr[dev] = p;
    }
    *out = addr[dev];
    return QMM_OK;
}

int qmm_gemv_noalloc(uint32_t fmt, const void* W, const void* x, float* y, int64_t N, int64_t K,
                     int B) {
    qmm_init();
    int wf;
    bool bf16, q8;
    int rc = check_gemv_args(fmt, W, x, y, N, K, B, &wf, &bf16, &q8);
    if (rc) return rc;
    if (is_kquant(wf)) return fail(QMM_EUNSUPPORTED, "qmm_gemv_noalloc supports q6_K, Q4_0 and Q8_0 weights");
    DevInfo* d;
    if ((rc = dev_info(&d))) return rc;
    GemvPlan p;
    if ((rc = plan_gemv(wf, q8, bf16, B, N, K, d->sms, &p))) return rc;
    if (p.ws_total > QMM_NOALLOC_SCRATCH_BYTES)
        return fail(QMM_ENOWORKSPACE,
                    "qmm_gemv_noalloc: this shape needs %zu bytes of scratch, the fixed array "
                    "holds %u",
                    p.ws_total, QMM_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch))) return rc;
    return run_gemv(wf, q8, bf16, W, x, y, N, K, B, p, static_cast<uint8_t*>(scratch), d);
}

int qmm_wait_probe(uint32_t limit_us) {
    qmm_init();
    if (limit_us < 1 || limit_us > 1000000)
        return fail(QMM_EINVAL, "limit_us = %u outside 1..1000000", limit_us);
    DevInfo* d;
    int rc = dev_info(&d);
    if (rc) return rc;
    cudaError_t e = wait_probe_launch(static_cast<unsigned long long>(limit_us) * 1000ull, t_stream, d->st);
    if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
    return QMM_OK;
}

const char* qmm_last_error(void) { return t_err; }

}  // extern "C"
