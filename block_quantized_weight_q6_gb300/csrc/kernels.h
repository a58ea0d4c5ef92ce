// kernels.h -- internal interface between the host dispatch (api.cu) and the
// kernel translation units. Not part of the public C interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qmm.h"

namespace qmm {

// ---------------------------------------------------------------- CUDA-core matvec pieces
// The routed-expert kernels (moe.cu) stream weight rows per warp: a warp owns
// (row group, K range) items, copies each chunk of CB consecutive blocks of
// its rows into a private ring of shared-memory slots with 1-D bulk TMA
// copies, and decodes them there (gemv_impl.cuh).
constexpr int kGemvWarps = 12;
constexpr int kGemvThreads = kGemvWarps * 32;

struct GemvArgs {
    const uint8_t* W;
    int64_t N, K, nb;      // rows, columns, blocks per row
    int64_t total_bytes;   // bytes of W (N * nb * block bytes)
    const void* x;         // float mode: [B][K] fp32 or bf16
    int x_bf16;
    const float* xf;       // float mode, many batch rows: the same activations as fp32
    const int8_t* xq;      // q8 mode: [B][K] int8
    const float* xs;       // q8 mode: [B][K/32] fp32
    int B;
    float* y;              // [B][N] when splits == 1
    float* part;           // [splits][B][N] when splits > 1
    int splits, cps, nchunks;
    int64_t n_items;       // ceil(N / R) * splits
    DevState st;
    int live_slot;
};

cudaError_t splitk_reduce_launch(const float* part, float* y, int splits, int64_t count,
                                 cudaStream_t s, DevState st);
// the split matrices of a grouped matvec, reduced in one launch (same order)
constexpr int kReduceSetMax = 12;
struct SplitReduceSet {
    const float* part[kReduceSetMax];
    float* y[kReduceSetMax];
    int64_t count[kReduceSetMax];  // B * N
    int64_t start[kReduceSetMax];  // first element of each matrix in the set
    int splits[kReduceSetMax];
    int n;
    int64_t total;
};
cudaError_t splitk_reduce_set_launch(const SplitReduceSet& r, cudaStream_t s, DevState st);

// ---------------------------------------------------------------- batch-1 matvec
// One activation row, float mode, on the CUDA cores (mv1.cuh): work item =
// block of kMv1RowBlock rows of one matrix, all of its K. Matrices of one
// launch share the format; K % 256 == 0.
constexpr int kMv1RowBlock = 4;
struct Mv1Mat {
    const uint8_t* W;
    const void* x;   // [B][K] fp32 or bf16
    float* y;        // [B][N]
    int64_t N, K, rowbytes;
    int pieces, full_pieces;  // K in the kernel's pieces (2048 for mv1, 256 for mv8), partial one included / not
    int aligned;              // W and the row pitch are 16-byte multiples
    int item0;                // first item of this matrix in the launch
};
struct Mv1Group {
    Mv1Mat m[12];
    int nmat, items;
    int x_bf16;
    int B;                    // activation rows (mv8: 2..8)
    int ks;                   // mv8: warps that share an item (1, 2, 4 or 8)
    DevState st;
    int live_slot;
};
// whether mv1 takes this (format, K) and resident CTAs per SM; launch
bool mv1_supported(int fmt, int64_t K);
int mv1_occupancy(int fmt);
cudaError_t mv1_launch(int fmt, int grid, cudaStream_t s, const Mv1Group& g);

// ---------------------------------------------------------------- batch 2-8 matvec
// 2..8 bf16 activation rows, float mode, on the warp-level MMA (mv8.cuh):
// work item = block of kMv8RowBlock rows of one matrix, all of its K, in
// stages of 256 K. The same group description as mv1 (pieces = K / 256,
// items of kMv8RowBlock rows); K % 256 == 0.
constexpr int kMv8RowBlock = 32;
bool mv8_supported(int fmt, int64_t K);
int mv8_occupancy(int fmt);
cudaError_t mv8_launch(int fmt, int grid, cudaStream_t s, const Mv1Group& g);

// ---------------------------------------------------------------- batch 1-8 fp16-MMA matvec
// 1..8 bf16 activation rows, float mode, any mix of the three formats in one
// launch, on the warp-level MMA with fp16 operands (mvh.cuh): work item = 16
// rows of one matrix at stride 8, all of its K. Needs K % 256 == 0 and
// N % 8 == 0, and workspace for the fp16 activations (mvh_workspace_bytes).
constexpr int kMvhWarps = 16;
constexpr int kMvhMaxMats = 12;
struct MvhMat {
    const uint8_t* W;
    const uint16_t* xh;   // the activations as fp16 x * 2^e per batch row, [B][K]
    const float* xinv;    // 2^-e per batch row
    float* y;             // [B][N]
    int64_t N, K, rowbytes;
    int fmt, stages, item0;
    int stage_bytes, stage_k, box_w, boxes;  // the format's stage shape, set by the host
};
struct MvhGroup {
    CUtensorMap map[kMvhMaxMats];  // W as [N / 8][8 * rowbytes] 16-bit elements, boxes 32 rows high
    MvhMat m[kMvhMaxMats];
    int* ctr;             // the next unclaimed item past the first wave (reset by the prep kernel)
    int nmat, items, B, ks;
    DevState st;
    int live_slot;
};
bool mvh_supported(int fmt, int64_t N, int64_t K);
// workspace for n matvecs whose activations are x[i] (equal pointers and K share it)
size_t mvh_workspace_bytes(int n, const void* const* x, const int64_t* K, int B);
// the prep kernel (bf16 -> scaled fp16) and the matvec over matrices
// sel[0 .. n-1] of the arrays, formats fmt[]
cudaError_t mvh_run(int n, const int* sel, const int* fmt, const void* const* W, const void* const* x,
                    float* const* y, const int64_t* N, const int64_t* K, int B, void* ws, int sms,
                    cudaStream_t s, DevState st);

// The routed-expert matvecs on the same kernel (mvh.cu): the tasks (expert,
// first grouped slot, tokens) come from moe.cu's plan kernel; an expert
// table is one tensor map with the expert as its third coordinate, so the
// experts of a table must lie at one fixed stride.
struct MoeTask {
    int expert, pos, n;  // expert, first grouped slot, tokens
};
struct MvhMoeTables {
    const void* base[3];   // gate, up, down of expert 0
    int64_t stride[3];     // bytes from one expert's matrix to the next
};
// rows a task of the fp16-MMA expert matvec holds (tokens per task)
constexpr int kMoeMvhTask = 4;
size_t moe_mvh_workspace_bytes(int T, int k, int H, int I);
// gate/up matvec, silu(g) * u, down matvec, over the plan in ws (see moe.cu)
cudaError_t moe_mvh_run(int fmt, int E, int H, int I, int T, int k, const MvhMoeTables& tab, const void* x,
                        const int* n_tasks, const MoeTask* tasks, const int* pos_slot, void* ws, float* o,
                        int sms, cudaStream_t s, DevState st);
bool moe_mvh_supported(int fmt, int H, int I);
// QMM_MOE_MMA=0 (read once by qmm_init) keeps moe_gemv on the CUDA-core expert matvec
extern bool g_moe_mvh_enabled;

// ---------------------------------------------------------------- tensor-core matvec
// Work item = (128-row tile, range of 256-wide K stages); see tcmv.cuh.
constexpr int kTcThreads = 768;
struct TcmvArgs {
    const uint8_t* W;
    int64_t N, K, nb;      // rows, columns, blocks per row
    int64_t total_bytes;   // bytes of W
    int64_t rowbytes;      // bytes per row
    int64_t n8;            // rows reached through the tensor map: 8 * floor(N / 8)
    const void* x;         // the activations [B][K] as given
    int x_bf16;            //   ... bf16 (else fp32); bf16 float mode gathers them in the matvec
    const uint16_t* xt;    // q8 and fp32 float mode: the prepared activation operand (tcmv.cu)
    const float* xs;       // q8 mode: activation scales [K / 32 rounded to stages][NB]
    int B;
    float* y;              // [B][N] when pieces == 1
    float* part;           // [pieces][B][N] when pieces > 1
    int64_t tiles, nst, sps, pieces, items;  // items = tiles * pieces
    int64_t item0;         // in a group: the first item of this matrix
    DevState st;
    int live_slot;
};

// One matvec launch over up to kTcMaxMats matrices of one format and batch:
// the items of matrix m are item0 .. item0 + items - 1 of the launch, in
// matrix order; map[m] is matrix m's weight tensor map (tcmv.cu).
constexpr int kTcMaxMats = 12;
struct TcmvGroup {
    CUtensorMap map[kTcMaxMats];
    TcmvArgs m[kTcMaxMats];
    int nmat;
    int64_t items;
    DevState st;
    int live_slot;
};

using TcmvKernel = void (*)(const TcmvGroup);

// cuTensorMapEncodeTiled through the runtime's driver entry point (null if
// the driver has none)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
TcmvKernel tcmv_pick_q6k(bool q8, int NB, int S);
TcmvKernel tcmv_pick_q4_0(bool q8, int NB, int S);
TcmvKernel tcmv_pick_q8_0(bool q8, int NB, int S);
uint32_t tcmv_smem_q6k(int NB, int S);
uint32_t tcmv_smem_q4_0(int NB, int S);
uint32_t tcmv_smem_q8_0(int NB, int S);

// MMA columns for NB activation rows split S ways (the matvec's NCOL)
inline int tcmv_ncol(int NB, int S) {
    const int nc = NB * S;
    return (nc >= 6 && nc <= 8) ? 64 : (nc >= 4 && nc <= 5) ? 32 : (nc <= 16 ? 16 : (nc <= 32 ? 32 : 48));
}
inline int tcmv_stage_blocks(int fmt) { return fmt == FMT_Q6_K ? 1 : 8; }
// resident CTAs per SM of the (fmt, q8, NB, S) kernel (0 if not built)
int tcmv_occupancy(int fmt, bool q8, int NB, int S);
// builds the weights' tensor map (W seen as rows of 8 weight rows) and launches
cudaError_t tcmv_launch(int fmt, bool q8, int NB, int S, int grid, cudaStream_t s,
                        const TcmvArgs& a);
// the same for a group (g.m[0 .. nmat-1], items and item0 filled in; the
// maps are filled here)
cudaError_t tcmv_launch_group(int fmt, bool q8, int NB, int S, int grid, cudaStream_t s, TcmvGroup& g);
// activations [B][K] (fp32 or bf16) -> the matvec's bf16 activation operand
// for weight format fmt (tcmv.cu); q8 mode quantizes per 32 first and also
// writes the scales as [block][NB]
cudaError_t act_tile_launch(const void* x, int x_bf16, int B, int64_t K, int fmt, int NB, int S,
                            int ncol, int64_t nst, bool q8, uint16_t* xt, float* xs, cudaStream_t s,
                            DevState st);
// the same for the matrices of a grouped matvec, in one launch
struct ActTileSet {
    const void* x[kTcMaxMats];
    int64_t K[kTcMaxMats];
    uint16_t* xt[kTcMaxMats];
    float* xs[kTcMaxMats];
    int64_t start[kTcMaxMats];  // first unit (16 bytes of operand) of each matrix
    int n, x_bf16, B, fmt, NB, S, ncol, q8;
    int64_t total;
};
cudaError_t act_tile_set_launch(const ActTileSet& r, cudaStream_t s, DevState st);

// one warp that waits on an mbarrier nothing completes, giving up after
// limit_ns (test aid for the bounded waits; tcmv.cu)
cudaError_t wait_probe_launch(unsigned long long limit_ns, cudaStream_t s, DevState st);

// ---------------------------------------------------------------- quantizer
// x [rows][K] (fp32 or bf16) -> xq [rows][K] int8, xs [rows][K/32] fp32.
// If a16 != nullptr, also writes the quantized values as fp16 in the GEMM's
// A-operand tile layout (see gemm.cu), for rows rounded up to 128.
cudaError_t quantize_q8_launch(const void* x, int x_bf16, int64_t rows, int64_t K, int8_t* xq,
                               float* xs, uint16_t* a16, cudaStream_t s, DevState st);

// ---------------------------------------------------------------- GEMM
// bytes of the fp16 A-operand tiles for M x K activations (M rounded up to 128)
size_t gemm_a16_bytes(int64_t M, int64_t K);
// K splits of an M x N x K GEMM (1 when its tiles fill the SMs), and the
// bytes of the split partials gemm_launch then needs (0 for one split)
int gemm_splits(int64_t M, int64_t N, int64_t K);
size_t gemm_part_bytes(int64_t M, int64_t N, int64_t K);
// fmt FMT_Q6_K (exp: plane variant) or FMT_Q4_0 (exp false); part: device
// workspace of gemm_part_bytes(M, N, K) bytes (null when that is 0)
cudaError_t gemm_launch(int fmt, bool exp, const uint8_t* W, const int8_t* plane,
                        const uint16_t* a16, const float* xs, float* Y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s, DevState st, int live_slot, float* part);

// One GEMM over several experts' rows: 128-row tile mt of A (M % 128 == 0)
// and Y belongs to expert tile_expert[mt] (device array), whose weights are
// W + expert * wstride (wstride % 16 == 0); fmt FMT_Q6_K or FMT_Q4_0, the
// in-kernel expansion, no K split.
cudaError_t gemm_grouped_launch(int fmt, const uint8_t* W, int64_t wstride, int n_experts, const int* tile_expert,
                                const uint16_t* a16, const float* xs, float* Y, int64_t M, int64_t N, int64_t K,
                                cudaStream_t s, DevState st, int live_slot);

// ---------------------------------------------------------------- MoE prefill
// (moe_prefill.cu) the T*k routing slots ordered by expert, stable: counts
// [E], order [S] (slots by expert), pos [S] (each slot's row in that order)
cudaError_t moe_prefill_plan_launch(const int32_t* idx, int S, int E, int* counts, int* order, int* pos,
                                    cudaStream_t s, DevState st);
// Xg[r] = x row of token order[r] / k (rows of rowbytes, a multiple of 16)
cudaError_t moe_prefill_gather_launch(const void* x, int64_t rowbytes, const int* order, int k, int S, void* Xg,
                                      int sms, cudaStream_t s, DevState st);
// the padded layout of a grouped launch (expert e's rows from poff[e], a
// multiple of 128): pos_pad[slot], and prow[row] = slot (rows left at -1
// are padding)
cudaError_t moe_prefill_padmap_launch(const int32_t* idx, const int* pos, const int* off, const int* poff, int S,
                                      int* pos_pad, int* prow, int sms, cudaStream_t s, DevState st);
// padded row r of Xg = x row of slot prow[r] / k, or zeros
cudaError_t moe_prefill_gather_pad_launch(const void* x, int64_t rowbytes, const int* prow, int k, int rows, void* Xg,
                                          int sms, cudaStream_t s, DevState st);
// g <- silu(g) * u over n values (n % 4 == 0)
cudaError_t moe_prefill_silu_launch(float* g, const float* u, int64_t n, int sms, cudaStream_t s, DevState st);
// y[t] = sum_j gate[t][j] * O[pos[t][j]], j in order (H % 4 == 0)
cudaError_t moe_prefill_combine_launch(const float* O, const int* pos, const float* gate, int T, int k, int H,
                                       float* y, cudaStream_t s, DevState st);

// ---------------------------------------------------------------- additive codebooks
// (cbk.cu) partial-sum bytes of the launch, and the launch itself
size_t cbk_part_bytes(int M, int64_t N, int64_t K, int B);
size_t cbk_smem_bytes(int M, int B);
cudaError_t cbk_launch(int M, const uint8_t* codes, const uint16_t* books, const uint16_t* scales, const void* x,
                       int x_bf16, float* y, int64_t N, int64_t K, int B, float* part, int sms, cudaStream_t s,
                       DevState st);

// ---------------------------------------------------------------- MoE
constexpr int kMoeMaxExperts = 1024;
constexpr int kMoeMaxSlots = 1024;  // tokens x top_k per call
constexpr int QMM_LIVE_ROUTE_SLOT = QMM_LIVE_ROUTE;
constexpr int QMM_LIVE_MOE_GATE_UP_SLOT = QMM_LIVE_MOE_GATE_UP;
constexpr int QMM_LIVE_MOE_DOWN_SLOT = QMM_LIVE_MOE_DOWN;
constexpr int QMM_LIVE_MOE_COMBINE_SLOT = QMM_LIVE_MOE_COMBINE;
constexpr int QMM_LIVE_MOE_PLAN_SLOT = QMM_LIVE_MOE_PLAN;
constexpr int QMM_LIVE_MOE_GATHER_SLOT = QMM_LIVE_MOE_GATHER;
size_t moe_workspace_bytes(int T, int k, int H, int I, bool x_bf16);
cudaError_t moe_launch(int fmt, int E, int H, int I, int T, int k, const void* const* wg,
                       const void* const* wu, const void* const* wd, const int32_t* idx,
                       const float* gate, const void* x, int x_bf16, float* y, void* ws, int sms,
                       cudaStream_t s, DevState st);
cudaError_t route_launch(const float* logits, int T, int E, int k, int32_t* idx, float* gate,
                         cudaStream_t s, DevState st);

// ---------------------------------------------------------------- plane
cudaError_t plane_build_launch(const uint8_t* W, int64_t N, int64_t K, int8_t* plane,
                               cudaStream_t s, DevState st);

}  // namespace qmm
