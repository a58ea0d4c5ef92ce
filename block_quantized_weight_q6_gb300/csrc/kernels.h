// kernels.h -- internal interface between the host dispatch (api.cu) and the
// kernel translation units. Not part of the public C interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "qmm.h"

namespace qmm {

// ---------------------------------------------------------------- GEMV
// One warp owns a run of (row group, K split) items; each item is R
// consecutive rows over a range of K chunks. A chunk is CB consecutive
// blocks of a row (q6_K: 8 super-blocks, Q4_0 / Q8_0: 32 blocks). The warp
// streams its chunks into a private ring of shared-memory slots with 1-D
// bulk TMA copies and decodes them from there.
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

using GemvKernel = void (*)(const GemvArgs);
GemvKernel gemv_pick_q6k(bool q8, int NB, int R);
GemvKernel gemv_pick_q4_0(bool q8, int NB, int R);
GemvKernel gemv_pick_q8_0(bool q8, int NB, int R);

// rows per item the variants prefer when N is large enough
inline int gemv_preferred_rows(bool q8, int NB) {
    (void)q8;
    (void)NB;
    return 4;
}
// whether the (mode, NB) variant reads its activations from the fp32 copy
// a.xf (the narrow, many-batch-row float variants)
inline bool gemv_needs_xf(bool q8, int NB, int R) {
    (void)R;
    return !q8 && NB >= 4;
}

// shared memory bytes of one CTA of the (fmt, R) kernel
size_t gemv_smem_bytes(int fmt, int R);
int gemv_chunk_blocks(int fmt);
// launches the kernel instantiation for (fmt, q8, NB, R); returns
// cudaErrorInvalidValue if that instantiation is not built.
cudaError_t gemv_launch(int fmt, bool q8, int NB, int R, int grid, cudaStream_t s,
                        const GemvArgs& a);
// max resident CTAs per SM for (fmt, q8, NB, R) (0 if not built)
int gemv_occupancy(int fmt, bool q8, int NB, int R);

// bf16 [n] -> fp32 [n]
cudaError_t x_to_f32_launch(const void* x_bf16, float* out, int64_t n, cudaStream_t s,
                            DevState st);

cudaError_t splitk_reduce_launch(const float* part, float* y, int splits, int64_t count,
                                 cudaStream_t s, DevState st);

// ---------------------------------------------------------------- quantizer
// x [rows][K] (fp32 or bf16) -> xq [rows][K] int8, xs [rows][K/32] fp32.
// If a16 != nullptr, also writes the quantized values as fp16 in the GEMM's
// A-operand tile layout (see gemm.cu), for rows rounded up to 128.
cudaError_t quantize_q8_launch(const void* x, int x_bf16, int64_t rows, int64_t K, int8_t* xq,
                               float* xs, uint16_t* a16, cudaStream_t s, DevState st);

// ---------------------------------------------------------------- GEMM
// bytes of the fp16 A-operand tiles for M x K activations (M rounded up to 128)
size_t gemm_a16_bytes(int64_t M, int64_t K);
// fmt FMT_Q6_K (exp: plane variant) or FMT_Q4_0 (exp false)
cudaError_t gemm_launch(int fmt, bool exp, const uint8_t* W, const int8_t* plane,
                        const uint16_t* a16, const float* xs, float* Y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s, DevState st, int live_slot,
                        float* dbg = nullptr);

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
