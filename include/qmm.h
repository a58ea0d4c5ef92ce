/*
 * qmm.h -- C interface of libqmm, matrix multiplication against
 * block-quantized LLM weights with the dequantization fused into the kernels,
 * written for NVIDIA GB300 (sm_103a).
 *
 * Conventions that hold for every call below unless its comment says
 * otherwise:
 *  - Pointers named W, x, X, y, Y, plane, idx, gate_w, logits are DEVICE
 *    pointers. The caller allocates and owns them (typically torch tensors);
 *    the library never frees them and keeps no reference after the call
 *    returns, except the plane registry described at qmm_plane_build.
 *  - Calls are asynchronous on the calling thread's current stream
 *    (qmm_set_stream); none synchronizes the device except
 *    qmm_liveness_read and qmm_sync_check.
 *  - Every call returns QMM_OK (0) or a negative QMM_E* code. Argument errors
 *    are detected on the host before anything is launched; qmm_last_error()
 *    then gives a one-line reason (thread-local, valid until the next call).
 *  - Weight matrices are row-major by output row n: row n is K/E consecutive
 *    blocks (E = 256 for q6_K, 32 for Q4_0 and Q8_0), with no padding between
 *    rows. W must be 16-byte aligned.
 *
 * Block formats (weight w of element i of a block; d is fp16 little-endian):
 *  q6_K, 210 B per 256 weights: ql[128] | qh[64] | scales[16] int8 | d.
 *      q = ((ql[i%128] >> 4*(i/128)) & 0xF) | ((qh[i%64] >> 2*(i/64)) & 3) << 4,
 *      w = d * scales[i/16] * (q - 32).  The element expansion is the one of
 *      "57 - r54 MINFER_MMQ_Q6K_EXP" section 2.1 (per 16-element group); the
 *      nibble order within ql/qh is this library's reading, stated here.
 *  Q4_0, 18 B per 32 weights: d | qs[16]; q = (qs[i%16] >> 4*(i/16)) & 0xF,
 *      w = d * (q - 8).
 *  Q8_0, 34 B per 32 weights: d | qs[32] int8; w = d * qs[i].
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* fmt = weight format | activation element type | activation mode */
enum {
    QMM_Q4_0 = 0x01,
    QMM_Q8_0 = 0x02,
    QMM_Q6_K = 0x03,
    /* The K-quant ladder formats of quantprobe "LAWS.md", Law 4 amendment
     * L-16 (a scale and a min per 32 weights for Q4_K, per 16 for Q2_K;
     * weight = d * scale_j * q - dmin * min_j). The pages give no byte
     * layout; the one read here, per 256-weight super-block:
     *   Q4_K, 144 B: d (fp16) | dmin (fp16) | 12 bytes of eight 6-bit scales
     *     and mins (sub-block j < 4: scale = b[j] & 63, min = b[j+4] & 63;
     *     j >= 4: scale = (b[j+4] & 15) | (b[j-4] >> 6) << 4, min =
     *     (b[j+4] >> 4) | (b[j] >> 6) << 4) | 128 code bytes; element i is
     *     nibble (i/32) % 2 (0 = low) of code byte 32 (i/64) + i % 32.
     *   Q2_K, 84 B: 16 bytes (sub-block i/16: low nibble scale, high nibble
     *     min) | 64 code bytes | d (fp16) | dmin (fp16); element i is the
     *     2-bit field at bit 2 ((i % 128) / 32) of code byte
     *     32 (i/128) + i % 32.
     * Rows are K/256 consecutive super-blocks. Only the matvecs take them
     * (qmm_gemv, qmm_gemv_group, qmm_gemv_multi and their workspace queries),
     * with bf16 activations in float mode, B <= 8, K % 256 == 0 and
     * N % 8 == 0; every other call refuses them with QMM_EUNSUPPORTED. */
    QMM_Q4_K = 0x04,
    QMM_Q2_K = 0x05,
    QMM_FMT_MASK = 0xFF,

    QMM_X_F32 = 0x000,  /* activations are fp32                              */
    QMM_X_BF16 = 0x100, /* activations are bfloat16                          */
    QMM_X_MASK = 0xF00,

    QMM_ACT_FLOAT = 0x0000, /* fp32 arithmetic on the activations as given    */
    QMM_ACT_Q8 = 0x1000,    /* activations quantized per 32 to int8 + fp32
                               scale (s = amax/127, x_q = round-half-even(x/s)),
                               then exact integer dot products per weight
                               group, as in quantprobe "LAWS.md" Law 4
                               amendment L-15 (dp4a matvec)                   */
    QMM_ACT_MASK = 0xF000
};

enum {
    QMM_OK = 0,
    QMM_EINVAL = -1,           /* null pointer, non-positive size, bad B/fmt  */
    QMM_EUNSUPPORTED = -2,     /* format/mode combination not built            */
    QMM_EALIGN = -3,           /* K not a multiple of the block, or a pointer
                                  not 16-byte aligned                          */
    QMM_ECUDA = -4,            /* a CUDA runtime call failed                   */
    QMM_EPLANE = -5,           /* exp_plane was not built for this W / N / K   */
    QMM_EDEVICE_TIMEOUT = -6,  /* a kernel gave up a bounded wait (see
                                  qmm_sync_check)                              */
    QMM_ENOWORKSPACE = -7      /* the call needs more workspace than is set    */
};

/* Liveness counters: one slot per kernel path, incremented once per launch by
 * the launched kernel itself (so a launch that silently never ran is not
 * counted). The four q6_K GEMM slots are the four labels of
 * "57 - r54 MINFER_MMQ_Q6K_EXP" section 3.2: plane path, raw weights that
 * never had a plane, plane deliberately switched off, plane expected but
 * missing (an accidental fallback). */
enum {
    QMM_LIVE_GEMV_FLOAT = 0,
    QMM_LIVE_GEMV_Q8 = 1,
    QMM_LIVE_GEMV_SPLITK_REDUCE = 2,
    QMM_LIVE_QUANTIZE = 3,
    QMM_LIVE_PLANE_BUILD = 4,
    QMM_LIVE_GEMM_EXP_PLANE = 5,      /* "W_exp-cp.async"                    */
    QMM_LIVE_GEMM_IN_KERNEL = 6,      /* "in-kernel-expand" (never eligible) */
    QMM_LIVE_GEMM_EXP_OFF = 7,        /* "in-kernel-expand(exp=off)"         */
    QMM_LIVE_GEMM_FALLBACK = 8,       /* "in-kernel-expand(fallback!)"       */
    QMM_LIVE_GEMM_Q4_0 = 9,
    QMM_LIVE_ROUTE = 10,
    QMM_LIVE_MOE_GATE_UP = 11,
    QMM_LIVE_MOE_DOWN = 12,
    QMM_LIVE_MOE_COMBINE = 13,
    QMM_LIVE_X_TILE = 14,             /* activations laid out as the matvec's
                                         tensor-core operand                 */
    QMM_LIVE_MOE_PLAN = 15,
    QMM_LIVE_MOE_GATHER = 16,
    QMM_LIVE_GEMV_MV1 = 17,           /* batch-1 float matvec on the CUDA
                                         cores                               */
    QMM_LIVE_GEMV_MV8 = 18,           /* batch 1-8 float matvec on the
                                         warp-level MMA (fp16 or bf16)       */
    QMM_LIVE_MOE_SILU = 19,           /* silu(g) * u laid out for the expert
                                         matvecs on the warp-level MMA       */
    QMM_LIVE_GEMM_SPLIT_REDUCE = 20,  /* sum of a GEMM's K-split partials
                                         (grids with fewer tiles than SMs)   */
    QMM_LIVE_MOE_PREFILL_PLAN = 21,   /* moe_prefill: slots ordered by
                                         expert, and (grouped flow) the
                                         padded row map                      */
    QMM_LIVE_MOE_PREFILL_ROWS = 22,   /* moe_prefill: activation rows
                                         gathered by expert, and the gated
                                         sum scattered back (two launches)   */
    QMM_LIVE_MOE_PREFILL_SILU = 23,   /* moe_prefill: silu(g) * u            */
    QMM_LIVE_CBK_GEMV = 24,           /* qmm_cbk_gemv: the table-lookup
                                         launch and its fixed-order sum      */
    QMM_LIVE_COUNT = 32
};

/* Reads the environment once: QMM_Q6K_EXP ("0" opts out of building W_exp
 * planes; unset or anything else keeps them on, the default-on / "0" opt-out
 * gate of "57 - r54 MINFER_MMQ_Q6K_EXP" section 3.1), QMM_DEBUG_LABEL ("1"
 * prints one stderr line per q6_K GEMM launch naming its path, section 2.4),
 * QMM_FAULT ("plane_alloc" makes qmm_plane_wanted's caller-side allocation be
 * treated as failed; host-side fault injection only), QMM_MV1 ("0" sends
 * batch-1 float matvecs to the tensor-memory matvec instead of the CUDA-core
 * one), QMM_MV8 ("0" does the same for the bf16 warp-level MMA matvec at
 * batch 2-8), QMM_MVH ("0" turns the fp16-MMA matvec for bf16 batches 1-8
 * off, so those batches take the paths above), QMM_PDL ("0" launches
 * without programmatic dependent launch), QMM_MOE_MMA ("0" keeps moe_gemv on
 * the CUDA-core expert matvec even where the warp-level MMA one applies),
 * QMM_MOE_GROUPED ("0" keeps moe_prefill on one GEMM launch per expert even
 * where the grouped launch applies).
 * Called implicitly by every entry point; calling it again is a no-op. */
int qmm_init(void);

/* Sets the CUDA stream (a cudaStream_t, e.g. torch's current stream) that the
 * calling thread's subsequent calls launch on. NULL selects the legacy
 * default stream. */
int qmm_set_stream(void* cuda_stream);

/* Sets the calling thread's workspace: a device buffer of `bytes` bytes,
 * 256-byte aligned, owned by the caller, that calls may use as scratch
 * (split-K partial sums, quantized activations, MoE intermediates). Calls on
 * the same stream may reuse it back to back; the caller must not use it
 * concurrently on two streams. */
int qmm_set_workspace(void* dev, size_t bytes);

/* Workspace that qmm_gemv (M_or_B = B) or qmm_gemm (M_or_B = M) needs for
 * these sizes; 0 if none. */
size_t qmm_workspace_bytes(uint32_t fmt, int64_t M_or_B, int64_t N, int64_t K);

/* Batched decode matvec, y[b][n] = sum_k w[n][k] * x[b][k], b < B <= 16:
 * the fused dequantize-and-multiply of quantprobe "LAWS.md", Law 4 and its
 * amendment L-15 (decode reads every weight once per token; the format's
 * unpack work, not its bit width, sets the cost).
 * x: [B][K] fp32 or bf16 (fmt bits), y: [B][N] fp32 (overwritten).
 * QMM_ACT_FLOAT: fp32 products and sums of the activations as given.
 * QMM_ACT_Q8: x is first quantized per 32 (needs workspace), then
 *   y = sum_g s_x * d * sc_g * I_g with exact int32 group partials I_g.
 * Float mode, K % 256 == 0: bf16 x with B = 1..8 and N % 8 == 0 runs on the
 * warp-level MMA with fp16 operands (x laid out once as fp16 scaled by a
 * power of two per row, in workspace; K split over the warps of a CTA for
 * short N, added in a fixed order); otherwise fp32 x at B = 1 with rows of
 * whole 16-byte pieces (q6_K K % 2048 == 0) runs on the CUDA cores, and bf16
 * x at B = 2..8 on the bf16 warp-level MMA (neither uses workspace). Every
 * other case runs on the tensor-memory matvec, where short N is split along
 * K and the partial sums are added in a fixed order by a second launch.
 * Either way the order of the sums is fixed, so results are bitwise
 * reproducible. */
int qmm_gemv(uint32_t fmt, const void* W, const void* x, float* y, int64_t N,
             int64_t K, int B);

/* Several decode matvecs in one launch: y[i] = W[i] x[i] for i < n <= 12,
 * each exactly as qmm_gemv(fmt, W[i], x[i], y[i], N[i], K[i], B) computes
 * it (the same format, activation type, mode and batch B for all). W, x, y,
 * N, K are host arrays of n entries; the pointers they hold are device
 * pointers with qmm_gemv's layouts and alignment. The launch walks the
 * 128-row tiles of all n matrices, so a short matrix does not leave the GPU
 * idle behind it (the 7B-shaped decode set runs as one call per format and
 * batch). Errors and workspace as qmm_gemv; the workspace size comes from
 * qmm_gemv_group_workspace_bytes. The split of K may differ from the single
 * call's, so results agree with qmm_gemv within the float bound, not
 * bitwise. */
int qmm_gemv_group(uint32_t fmt, int n, const void* const* W, const void* const* x,
                   float* const* y, const int64_t* N, const int64_t* K, int B);

/* Workspace that qmm_gemv_group needs for these shapes; 0 if none or if the
 * arguments are invalid. */
size_t qmm_gemv_group_workspace_bytes(uint32_t fmt, int n, const int64_t* N, const int64_t* K,
                                      int B);

/* Several decode matvecs whose weights may be of DIFFERENT formats, as one
 * call: y[i] = W[i] x[i] for i < n <= 12, each as qmm_gemv(fmt[i], W[i],
 * x[i], y[i], N[i], K[i], B) defines it (quantprobe "LAWS.md", Law 4: the
 * matvecs of one decode step read every weight once). All fmt[i] must share
 * the activation type and mode bits; the weight format bits may differ. In
 * float mode with bf16 activations, B <= 8, K % 256 == 0 and N % 8 == 0,
 * every matrix runs in ONE launch of the fp16-MMA matvec (after one launch
 * that lays the activations out), so a 7B-shaped decode step of mixed Q4_0 /
 * q6_K / Q8_0 weights is two launches; other matrices run per format as
 * qmm_gemv_group would run them. W, x, y, N, K, fmt are host arrays of n
 * entries (device pointers with qmm_gemv's layouts and alignment). Results
 * agree with qmm_gemv within the float bound (the order of the sums inside
 * a matrix may differ with the split of K). Workspace from
 * qmm_gemv_multi_workspace_bytes; errors as qmm_gemv. */
int qmm_gemv_multi(int n, const uint32_t* fmt, const void* const* W, const void* const* x,
                   float* const* y, const int64_t* N, const int64_t* K, int B);

/* Workspace that qmm_gemv_multi needs for these shapes (assuming no two
 * matvecs share their activations); 0 if none or if the arguments are
 * invalid. */
size_t qmm_gemv_multi_workspace_bytes(int n, const uint32_t* fmt, const int64_t* N, const int64_t* K,
                                      int B);

/* Size of the fixed scratch array that qmm_gemv_noalloc uses (4 MiB). */
#define QMM_NOALLOC_SCRATCH_BYTES (4u << 20)

/* The batched matvec of qmm_gemv (same arguments, same definition of y),
 * for callers that cannot allocate device memory when they call:
 * code hosted by an engine or framework that owns all device memory and
 * hands out only the input and output buffers, and latency-critical loops
 * that must not call into an allocator after start-up (cudaMalloc can block
 * on locks and synchronize the device). It needs no workspace: its scratch
 * (split-K partial sums, quantized or fp32 activation copies) lives in a
 * fixed array of QMM_NOALLOC_SCRATCH_BYTES that the library keeps in device
 * memory on every GPU that loads it, until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 * The first call on each device looks up that array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Shapes whose scratch would exceed the array are refused with
 * QMM_ENOWORKSPACE before anything is launched. Every call uses the same
 * array and leaves its contents behind (each call overwrites what it reads),
 * so two calls that run at the same time on the GPU (e.g. on two streams)
 * race: keep them ordered on one stream. It always runs the tensor-memory
 * matvec (the kernel that needs scratch), at every batch size, whereas
 * qmm_gemv sends float-mode batches of 1..8 with K % 256 == 0 to kernels
 * that use none; the two therefore agree within the float bound
 * |y - y'| <= 1e-4 * sum_k |w x| + 1e-6, not bitwise (q8 mode and the shapes
 * that qmm_gemv also sends to the tensor-memory matvec give the same bits).
 * The pages have no counterpart to this entry point. */
int qmm_gemv_noalloc(uint32_t fmt, const void* W, const void* x, float* y, int64_t N,
                     int64_t K, int B);

/* The per-32 activation quantizer on its own (the first step of QMM_ACT_Q8
 * and of qmm_gemm): x [rows][K] of type x_type (QMM_X_F32 or QMM_X_BF16),
 * K % 32 == 0 -> xq [rows][K] int8 and s [rows][K/32] fp32 with
 * s = amax/127 and xq = round-half-even(x/s) clamped to [-127, 127], both
 * divisions IEEE fp32; a block whose s is 0 gives zeros. x, xq 16-byte
 * aligned. */
int qmm_quantize_q8(uint32_t x_type, const void* x, int64_t rows, int64_t K, int8_t* xq,
                    float* s);

/* Prefill GEMM, Y[m][n] = sum_b s_x[m][b] * sum_{g in b} d[n] * sc[n][g] *
 * sum_{k in g} x_q[m][k] * c[n][k], with X quantized per 32 as in
 * QMM_ACT_Q8 and c the centered weight code. X: [M][K] bf16, Y: [M][N] fp32.
 * The integer partials run on the tensor cores (tcgen05, fp16 operands that
 * hold the integers exactly, fp32 accumulation that stays exact per 32-wide
 * block).
 * q6_K: exp_plane != NULL selects the W_exp-plane variant (the B tile is a
 *   plain copy of the centered-int8 plane, "57 - r54 MINFER_MMQ_Q6K_EXP"
 *   section 2.1, first bullet); NULL selects in-kernel ql/qh expansion
 *   (second bullet). The two give bitwise-identical Y (section 2.3). The
 *   plane must come from qmm_plane_build for this same W, N and K, else
 *   QMM_EPLANE.
 * Q4_0: in-kernel expansion only; exp_plane must be NULL.
 * Scales: any int8 q6_K sub-block scale. The fp16 B tile holds
 *   s * (q - 32) exactly for |s| <= 56, so a 128 x 128 output tile whose
 *   weights hold a larger scale sc runs its K range twice, with
 *   sc = s0 + 2 s1 (|s0| <= 56, |s1| <= 36, both of sc's sign), summing
 *   both passes; every block partial stays an exact integer.
 * Needs workspace (quantized X). */
int qmm_gemm(uint32_t fmt, const void* W, const void* X, float* Y, int64_t M,
             int64_t N, int64_t K, const int8_t* exp_plane);

/* Bytes of the W_exp plane of an N x K q6_K matrix: N*K (one centered int8
 * per weight, "57 - r54 MINFER_MMQ_Q6K_EXP" section 2.2). */
size_t qmm_plane_bytes(int64_t N, int64_t K);

/* Whether the registration gate builds a plane for an N x K q6_K matrix:
 * QMM_Q6K_EXP != "0" AND K % 256 == 0 (section 3.1, "AND semantics").
 * Returns 1 or 0. With QMM_FAULT=plane_alloc it still returns 1, and
 * qmm_plane_build(W, N, K, NULL) then records the failure. */
int qmm_plane_wanted(int64_t N, int64_t K);

/* Builds the plane of W into plane_dst (qmm_plane_bytes(N, K) bytes, device,
 * caller-owned) and registers it as W's plane: plane[n][k] = q(n,k) - 32.
 * plane_dst == NULL records that a plane was wanted for W but could not be
 * allocated; later qmm_gemm calls on W with a NULL plane are then counted as
 * QMM_LIVE_GEMM_FALLBACK, and "fallback!" is printed once to stderr
 * (section 1, failure semantics). */
int qmm_plane_build(const void* W_q6k, int64_t N, int64_t K, int8_t* plane_dst);

/* Forgets the registration of W's plane (call before freeing either). */
int qmm_plane_release(const void* W_q6k);

/* Routed experts of one MoE layer, all in format fmt, all resident in device
 * memory: w_gate[e], w_up[e] are inter x hidden, w_down[e] is hidden x inter.
 * The three pointer arrays are HOST arrays of n_experts DEVICE pointers. */
typedef struct {
    int n_experts, hidden, inter, top_k, n_tokens;
    const void* const* w_gate;
    const void* const* w_up;
    const void* const* w_down;
} qmm_moe_t;

/* Routed expert FFN for n_tokens tokens ("Chasing x100", section "Where the
 * wall actually fell: inversion": experts stay resident and are decoded in
 * place): for each token t and each of its top_k experts e = idx[t][j],
 * h = silu(Wg_e x_t) * (Wu_e x_t), o = Wd_e h, and
 * y[t] = sum_j gate_w[t][j] * o_j, summed in j order.
 * With bf16 x, hidden and inter multiples of 256, and each of the three
 * pointer tables at one fixed stride (w[e] = w[0] + e * stride, stride a
 * multiple of 16 bytes: experts allocated as one tensor), the expert
 * matvecs run on the warp-level MMA with fp16 operands (h enters the down
 * projection as two fp16 terms, 22 bits of its fp32 value); otherwise on the
 * CUDA cores. Either way each output is within the propagated float bound.
 * idx: [T][top_k] int32, gate_w: [T][top_k] fp32, x: [T][hidden] (fmt's
 * activation type), y: [T][hidden] fp32. Float activation mode only. Each
 * selected expert's matrices are read once per call however many of the
 * tokens chose it. Needs workspace. */
int moe_gemv(uint32_t fmt, const qmm_moe_t* experts, const int32_t* idx,
             const float* gate_w, const void* x, float* y);

/* Workspace moe_gemv needs. */
size_t qmm_moe_workspace_bytes(const qmm_moe_t* experts);

/* Expert-grouped MoE prefill (quantprobe "LAWS.md", L-30: prefill divides
 * parameters rather than bytes): the routed expert FFN of moe_gemv for a
 * prompt's tokens, with each expert's weights read once for all the tokens
 * that chose it. The T * top_k routing slots are ordered by expert (stable
 * in slot order), each expert's activation rows gathered into one matrix,
 * and g = Wg_e X_e, u = Wu_e X_e and o = Wd_e h_e computed by qmm_gemm's
 * prefill GEMM (activations quantized per 32, exact integer group
 * partials), with h = silu(g) * u in fp32 quantized per 32 again as the
 * down projection's input; y[t] = sum_j gate_w[t][j] * o_j, in j order.
 * Experts: q6_K or Q4_0 (the GEMM's formats), hidden and inter multiples of
 * 32 (256 for q6_K), each matrix 16-byte aligned (any address, no stride
 * needed). When each of w_gate, w_up and w_down lists its experts at one
 * fixed stride (a multiple of 16 bytes, at least one matrix), every
 * expert's rows are padded to whole 128-row tiles and each projection runs
 * as one grouped GEMM launch over all tiles (the tile's expert selects the
 * weights); any other table runs one GEMM per expert. The two flows meet
 * the same bound; their sums are grouped differently (the per-expert GEMMs
 * may split K), so their outputs can differ in the last bits. idx: [T][top_k] int32 device, gate_w: [T][top_k] fp32 device,
 * x: [T][hidden] fp32 or bf16 (fmt's activation type), y: [T][hidden] fp32;
 * x and y 16-byte aligned; T * top_k <= 2^22. Needs the workspace
 * qmm_moe_prefill_workspace_bytes gives. The call reads the per-expert
 * token counts back to the host (one stream synchronization) to size the
 * GEMMs, so it cannot be captured in a CUDA graph (QMM_EUNSUPPORTED while
 * the stream is capturing). An expert index outside 0..n_experts-1 returns
 * QMM_EINVAL after that synchronization (and sets the device flag
 * qmm_sync_check reports). Results are bitwise reproducible for a given
 * table layout. */
int moe_prefill(uint32_t fmt, const qmm_moe_t* experts, const int32_t* idx,
                const float* gate_w, const void* x, float* y);

/* Workspace moe_prefill needs (0 if the arguments are invalid). */
size_t qmm_moe_prefill_workspace_bytes(uint32_t fmt, const qmm_moe_t* experts);

/* Matvec against an additive-codebook matrix ("Chasing x100", "The kernel
 * is ready": the 2-bit and 3-bit additive codebook matvec). The pages give
 * no layout; the one read here: n_books (2 or 3) codebooks of 256 entries,
 * each 8 fp16 values, books[m][c][j] ([n_books][256][8] fp16, device);
 * codes[n][g][m], one byte per book for each group of 8 consecutive weights
 * of row n ([N][K/8][n_books] uint8, device); scales[n] one fp16 per row
 * (device). Weight 8g + j of row n is scale[n] * sum_m books[m][codes[n][g]
 * [m]][j], so a weight costs 2 (n_books = 2) or 3 bits plus the shared
 * books. y[b][n] = sum_k w[n][k] * x[b][k] for b < B <= 8; x: [B][K] of
 * x_type (QMM_X_F32 or QMM_X_BF16), y: [B][N] fp32 (overwritten). K % 128
 * == 0; codes, books, x 16-byte aligned. The kernel builds, per chunk of K,
 * the table of every book entry's dot with each 8-wide activation slice
 * (fp32) and sums table entries; chunk sums are added in a fixed order, so
 * results are bitwise reproducible and within 1e-4 * sum_k sum_m |scale *
 * book term * x| + 1e-6 of the exact product. Needs the workspace
 * qmm_cbk_workspace_bytes gives. */
int qmm_cbk_gemv(int n_books, const uint8_t* codes, const uint16_t* books, const uint16_t* scales,
                 uint32_t x_type, const void* x, float* y, int64_t N, int64_t K, int B);

/* Workspace qmm_cbk_gemv needs (0 if the arguments are invalid). */
size_t qmm_cbk_workspace_bytes(int n_books, int64_t N, int64_t K, int B);

/* Router helper: per token, the k largest of E fp32 logits (ties go to the
 * lower expert index) and their softmax over those k, the routing of the
 * 256-expert top-8 layer whose selected experts "Chasing x100" (section
 * "Where the wall actually fell: inversion") keeps resident and decodes in
 * place; softmax over the k selected logits, so the k gates sum to 1. logits: [T][E],
 * idx: [T][k] int32, gate_w: [T][k] fp32. E <= 1024, k <= 32. */
int qmm_route_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx,
                           float* gate_w);

/* Copies the first n liveness counters to the HOST array counts (synchronizes
 * the current device). */
int qmm_liveness_read(int64_t* counts, int n);
int qmm_liveness_reset(void);

/* Synchronizes the current stream and reports what kernels flagged since the
 * last check (the flags are cleared): QMM_EDEVICE_TIMEOUT if a kernel gave up
 * a bounded wait, QMM_EINVAL if moe_gemv met an expert index out of range. */
int qmm_sync_check(void);

/* Test aid for the bounded device waits: launches one warp that waits,
 * through the same warp-collective bounded wait as the tensor-memory matvec,
 * on an mbarrier that nothing ever completes. After limit_us microseconds
 * (1..1000000) the wait gives up and sets the timeout bit of the error word,
 * so the next qmm_sync_check returns QMM_EDEVICE_TIMEOUT (and clears it);
 * the kernel holds no copies or tensor memory, so the context stays usable.
 * The pages have no counterpart to this entry point. */
int qmm_wait_probe(uint32_t limit_us);

/* Reason for the calling thread's last non-OK return. */
const char* qmm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
