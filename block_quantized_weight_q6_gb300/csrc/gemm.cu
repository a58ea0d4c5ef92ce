// gemm.cu -- prefill GEMM against q6_K / Q4_0 weights on the sm_103a tensor
// cores (tcgen05, accumulators in tensor memory).
//
// Y[m][n] = sum_b s_x[m][b] * D[n][b] * I[m][n][b], b = 32-wide K blocks:
//   q6_K: I = sum_k x_q[m][k] * sc[n][k/16] * (q[n][k] - 32), D = d[n][k/256]
//   Q4_0: I = sum_k x_q[m][k] * (q[n][k] - 8),               D = d[n][b]
// The integer partials run on the tensor cores as an fp16 MMA: x_q (|.| <=
// 127) and sc*(q-32) (|.| <= 1024) are exact fp16 values, every product is an
// integer below 2^17 and a 32-wide block sums to below 2^22, so the fp32
// accumulator holds I exactly. The accumulator is drained once per K block
// and the scales are applied on the CUDA cores.
//
// Exactness of the B values: s * (q - 32) is formed as (off + c) * s -
// off * s with one rounding (off = 1056 from the raw bits, 1152 from the
// plane), so off * s must be a finite fp16 and the result an exact one:
// |s| <= kScMax = 56 keeps both (|s * (q - 32)| <= 1792). A q6_K sub-block
// scale sc (any int8) is split as sc = s0 + 2 s1 with s0 and s1 of sc's
// sign, |s0| <= 56 and |s1| <= 36 (|s0| = |sc| up to 56; beyond, 56 or 55,
// whichever leaves an even rest). The K loop runs with B = s0 * (q - 32);
// a CTA whose tile held a scale beyond 56 runs it a second time with B =
// s1 * (q - 32) and d doubled, summing both passes into the same outputs.
// Each pass's block partials stay exact integers. (The synthetic workloads
// draw sc on -32..31: one pass.)
//
// The two q6_K variants of "57 - r54 MINFER_MMQ_Q6K_EXP" section 2.1:
//   EXP  : the B tile comes from the centered-int8 W_exp plane (one byte per
//          weight, a plain copy; only the sub-block scale is applied);
//   !EXP : the B tile is expanded in the kernel from the raw ql / qh bytes.
// Both write exactly the same fp16 values into the B tile, and everything
// after that is shared code, so their outputs are bitwise identical (section
// 2.3: identity by construction).
//
// CTA roles (896 threads):
//   warp 0      A producer: 1-D bulk TMA copies of the A tiles (quantized
//               activations, pre-tiled by the quantizer), NS stages ahead
//               of the MMAs
//   warp 2      raw producer: the weight stages, up to NR 256-column chunks
//               ahead of the converters: q6_K / Q4_0 rows through a tensor
//               map (W as groups of 8 rows); the plane variant takes its
//               plane tile and each row's scales and d the same way
//   warp 1      owns the tensor memory; one lane issues tcgen05.mma, the
//               KP blocks of a stage into two of the NACC = 4 accumulator
//               buffers, and signals the epilogue once per stage
//   warps 4-11  converters: weights -> fp16 B tile (core-matrix layout);
//               warp cw converts the rows 8 g + cw (the plane variant:
//               g + 16 cw)
//   warps 12-27 epilogue: tcgen05.ld of the accumulators, scaling, output
//   warp 3      idle (it only joins the barrier at the end of each K pass)
// Registers are moved between warpgroups (setmaxnreg): the producers' and
// the MMA's warpgroup gives up most of its share to the epilogue's.
// Handing work between warps through an mbarrier costs a few hundred cycles
// of a warp's time, so the epilogue and the MMA meet once per stage of KP
// blocks rather than once per block.
#include <cuda_fp16.h>

#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"

namespace qmm {

namespace {

constexpr int BM = 128;           // tokens per tile (tensor-memory lanes)
constexpr int BN = 128;           // weight rows per tile (accumulator columns)
constexpr int KP = 2;             // K blocks (32 wide) per stage: one handoff per pair of blocks
constexpr int NS = 3;             // stages, each the A and B tiles of KP blocks
constexpr int kPrefetch = 8;      // stages of A tiles prefetched into L2 ahead of their copy
constexpr int kScMax = 56;        // largest |q6_K sub-block scale| the fp16 B tile holds exactly
constexpr int NR = 3;             // raw weight stages (256 columns each)
constexpr int NACC = 4;           // accumulator buffers in tensor memory: two stages of KP blocks
constexpr int DR_Q6K = 4;         // d ring depth, q6_K (per 256 columns)
constexpr int DR_Q40 = 16;        // d ring depth, Q4_0 (per 32 columns)
constexpr int kThreads = 896;                // 28 warps (7 warpgroups), 72 registers a thread at launch
constexpr int kRawWarp = 2;                 // raw weight producer
constexpr int kConv0 = 4, kConvWarps = 8;   // converter warps (warpgroups 1, 2)
constexpr int kConvRows = 8 / kConvWarps;   // rows 8 g + j a converter lane takes per pass (j = kConvRows cw + jj)
constexpr int kEpi0 = 12, kEpiWarps = 16;   // epilogue warps (warpgroups 3 .. 6)
constexpr int kEpiCols = BN * 4 / kEpiWarps;  // accumulator columns per epilogue thread
// registers per thread after the reallocation: 4 warps x 56 + 8 x 64 + 16 x 80 = 2016 x 32, the
// whole 28 x 72 x 32 the block is launched with (an increase beyond that pool would never
// complete). The producers' warpgroup needs its 56: with fewer it spills, and the slower
// issue of the raw-weight copies cost up to 12% of the GEMM (measured).
struct RegSplit {
    int low, conv, epi;
};
__host__ __device__ constexpr RegSplit reg_split(int, bool, bool = false) {
    return RegSplit{56, 64, 80};
}
static_assert(4 * reg_split(FMT_Q6_K, false).low + kConvWarps * reg_split(FMT_Q6_K, false).conv +
                      kEpiWarps * reg_split(FMT_Q6_K, false).epi <=
                  kThreads / 32 * 72,
              "register pool");
static_assert(kEpiCols == 32, "one 32-column tensor-memory load per block and thread");
constexpr int kTmemCols = 512;    // NACC * BN accumulators
constexpr int kATile = BM * 32 * 2;   // bytes of one A stage
// B stage: 16 groups of 8 weight rows, kBSbo bytes apart (a 16-byte odd
// multiple past 512, so that 8 lanes storing one row each of 8 different
// groups hit 8 different bank groups); core matrices 128 bytes apart along K
constexpr int kBSbo = 528;
constexpr int kBTile = 16 * kBSbo;    // bytes of one block's B tile
constexpr int kAStage = KP * kATile, kBStage = KP * kBTile;

// raw stage row strides (16-byte multiples with room for the lead-in)
constexpr int kRawQ6K = 240;      // one 210-byte super-block
constexpr int kRawQ40 = 176;      // up to 8 18-byte blocks
constexpr int kRawScale = 48;     // plane variant: a super-block's 16 scales and d with their lead-in
constexpr int kPlaneTile = 16 * BN * 16;  // plane variant: 256 columns of 128 rows, [16-column chunk][row][16]

struct SmemLayout {
    uint32_t a, b, raw, rawslot, dv, bars, tslot, abort_flag;
    uint32_t total;
};

// Raw stage of q6_K / Q4_0 rows (tensor-map layout): 8 boxes, box j holding
// row j of each of the tile's 16 groups of 8 rows at RS-byte slots, then a
// tail area for the up to 7 rows past the last whole group of 8 rows of W.
// A plane stage is the plane tile (16-byte column chunk c of row n at
// 2048 c + 16 n) followed by such a row area of kRawScale-byte slots that
// holds each row's scales and d.
__host__ __device__ constexpr uint32_t raw_slot_bytes(int rs, bool exp) {
    return (exp ? static_cast<uint32_t>(kPlaneTile) : 0u) + 8u * 16u * rs + 8u * rs;
}

__host__ __device__ constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int fmt, bool exp) {
    SmemLayout L{};
    const uint32_t rs = exp ? kRawScale : (fmt == FMT_Q6_K ? kRawQ6K : kRawQ40);
    const uint32_t dr = fmt == FMT_Q6_K ? DR_Q6K : DR_Q40;
    uint32_t o = 0;
    L.a = o;
    o += NS * kAStage;
    L.b = o;
    o += NS * kBStage;
    L.raw = o;
    L.rawslot = raw_slot_bytes(static_cast<int>(rs), exp);
    o += NR * L.rawslot;
    L.dv = o;
    o += dr * BN * 4;
    o = align_up(o, 8);
    L.bars = o;
    o += 8 * (2 * NS + 2 * NR + 2 * NACC + dr);
    L.tslot = o;
    o += 4;
    L.abort_flag = o;
    o += 4;
    L.total = align_up(o, 128);
    return L;
}

// barrier indices: full[NS] (the A copy's bytes and the converters),
// empty[NS], raw_full[NR], raw_empty[NR], acc_full[NACC], acc_empty[NACC]
// (one per accumulator buffer, i.e. per K block), dv_full[DR]
constexpr int NP = NACC;
__device__ __forceinline__ uint32_t bar_full(uint32_t B, int s) { return B + 8 * s; }
__device__ __forceinline__ uint32_t bar_empty(uint32_t B, int s) { return B + 8 * (NS + s); }
__device__ __forceinline__ uint32_t bar_raw_full(uint32_t B, int r) { return B + 8 * (2 * NS + r); }
__device__ __forceinline__ uint32_t bar_raw_empty(uint32_t B, int r) { return B + 8 * (2 * NS + NR + r); }
__device__ __forceinline__ uint32_t bar_acc_full(uint32_t B, int i) { return B + 8 * (2 * NS + 2 * NR + i); }
__device__ __forceinline__ uint32_t bar_acc_empty(uint32_t B, int i) {
    return B + 8 * (2 * NS + 2 * NR + NP + i);
}
__device__ __forceinline__ uint32_t bar_dv_full(uint32_t B, int i) {
    return B + 8 * (2 * NS + 2 * NR + 2 * NP + i);
}

// ---------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor, K-major operand without swizzle: core
// matrices of 8 rows x 16 bytes, adjacent along K 128 bytes apart (leading
// byte offset), adjacent 8-row groups 512 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo = 512) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((128u >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version of the sm_100 family
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4)                                 // D format fp32
           | (0u << 7) | (0u << 10)                  // A, B format fp16
           | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- trace
// Diagnostic builds define QMM_GEMM_TRACE and point qmm_gemm_trace at mapped
// host memory (128 words per CTA of a one-split grid): each warp records
// where it is, so a stall can be located from the host while the kernel is
// still running. Product builds compile it out.
#ifdef QMM_GEMM_TRACE
__device__ unsigned* qmm_gemm_trace;
#define QMM_TRACE(code, kb)                                                                   \
    do {                                                                                      \
        if (qmm_gemm_trace && (threadIdx.x & 31) == 0) {                                       \
            unsigned* t_ = qmm_gemm_trace + (blockIdx.y * gridDim.x + blockIdx.x) * 128 + 4 * (threadIdx.x >> 5); \
            asm volatile("st.volatile.global.u32 [%0], %1;" ::"l"(t_), "r"((unsigned)(code)) : "memory"); \
            asm volatile("st.volatile.global.u32 [%0], %1;" ::"l"(t_ + 1), "r"((unsigned)(kb)) : "memory"); \
        }                                                                                     \
    } while (0)
#else
#define QMM_TRACE(code, kb) \
    do {                    \
    } while (0)
#endif

// ---------------------------------------------------------------- waits

__device__ __forceinline__ bool aborted(uint32_t flag) { return lds_u32(flag) != 0; }

// try_wait that may suspend the thread (up to a 20 us hint, resuming when
// the phase completes) instead of spinning: the converter warps share the
// issue slots with every waiting role.
__device__ __forceinline__ bool mbar_wait_hint(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Bounded wait that also gives up once another role of the CTA has given up.
// Warp-collective: every lane of the calling warp polls (a converged warp
// resumes promptly from the suspending try_wait), and all lanes leave
// together with the same result, so the warp is converged afterwards (the
// tensor-memory loads and stores that follow are .sync.aligned).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint32_t flag,
                                              unsigned int* err) {
    if (__all_sync(0xffffffffu, mbar_wait_hint(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_wait_hint(bar, parity))) return true;
        if ((it & 3u) == 0) {
            int give_up = aborted(flag) ? 1 : 0;
            if (!give_up && globaltimer_ns() - t0 > kWaitLimitNs) give_up = 2;
            give_up = __shfl_sync(0xffffffffu, give_up, 0);
            if (give_up) {
                if (give_up == 2 && (threadIdx.x & 31) == 0) {
                    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(flag), "r"(1u) : "memory");
                    atomicOr(err, DERR_GEMM_TIMEOUT);
                }
                __syncwarp();
                return false;
            }
        }
    }
}


// ---------------------------------------------------------------- B tile
// Converter lane (kc = lane / 8, rw = lane % 8) writes 8 fp16 values: row
// n = 8 * rg + rw, columns 8 * kc .. + 7 of the 32-wide block, at
// rg * 512 + kc * 128 + rw * 16 (core-matrix layout; one warp store covers
// 512 contiguous bytes).

// code bytes (0..63, or 0..15) -> fp16 pairs (1024 + code)
__device__ __forceinline__ uint32_t half_pair_lo(uint32_t w) { return __byte_perm(w, 0x64646464u, 0x5140); }
__device__ __forceinline__ uint32_t half_pair_hi(uint32_t w) { return __byte_perm(w, 0x64646464u, 0x7362); }

// fma on fp16 pairs: a * b + c, rounded once
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t half2_bits(float x) {
    const uint32_t h = __half_as_ushort(__float2half_rn(x));
    return h | (h << 16);
}

// Bulk prefetch of global memory into L2 (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(addr));
}

// The 16 bytes at byte offset QW * 4 + sh / 8 of the 32 bytes w (sh 0, 8,
// 16 or 24): a funnel shift per word.
template <int QW>
__device__ __forceinline__ void pick16_at(const uint32_t (&w)[8], uint32_t sh, uint32_t (&o)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(w[QW + k], w[QW + k + 1], sh);
}

// The 16 bytes at byte offset off (0..15, the same in every lane of the
// warp) of the 32 bytes w: a warp-uniform branch on the word offset.
__device__ __forceinline__ void pick16(const uint32_t (&w)[8], uint32_t off, uint32_t (&o)[4]) {
    const uint32_t sh = (off & 3u) * 8u;
    switch (off >> 2) {
        case 0: pick16_at<0>(w, sh, o); break;
        case 1: pick16_at<1>(w, sh, o); break;
        case 2: pick16_at<2>(w, sh, o); break;
        default: pick16_at<3>(w, sh, o); break;
    }
}

// pick16 of four 32-byte runs at one offset, under one branch
__device__ __forceinline__ void pick16x4(const uint32_t (&w0)[8], const uint32_t (&w1)[8],
                                         const uint32_t (&w2)[8], const uint32_t (&w3)[8], uint32_t off,
                                         uint32_t (&o0)[4], uint32_t (&o1)[4], uint32_t (&o2)[4],
                                         uint32_t (&o3)[4]) {
    const uint32_t sh = (off & 3u) * 8u;
#define QMM_PICK4(QW)                \
    pick16_at<QW>(w0, sh, o0);      \
    pick16_at<QW>(w1, sh, o1);      \
    pick16_at<QW>(w2, sh, o2);      \
    pick16_at<QW>(w3, sh, o3);
    switch (off >> 2) {
        case 0: QMM_PICK4(0) break;
        case 1: QMM_PICK4(1) break;
        case 2: QMM_PICK4(2) break;
        default: QMM_PICK4(3) break;
    }
#undef QMM_PICK4
}

}  // namespace

// ---------------------------------------------------------------- kernel

struct GemmArgs {
    const uint8_t* W;      // q6_K or Q4_0 rows
    const int8_t* plane;   // W_exp plane (EXP variant)
    const uint16_t* a16;   // quantized activations as fp16, tiled
    const float* xs;       // [M][K/32] activation scales
    float* Y;              // [M][N]
    int64_t M, N, K, nb;   // nb: blocks per row
    int64_t total_bytes;   // bytes of W
    int64_t rowbytes;      // bytes per row of W
    int64_t n8;            // rows of W reached through the tensor map: 8 * floor(N / 8)
    int64_t kb_split;      // K blocks per split (a multiple of 8): CTA z takes blocks z * kb_split ..
    float* part;           // split partial outputs, split z at part + z * pstride as [M][N]; or
                           // null: the CTA writes Y
    int64_t pstride;       // floats per split: M * N rounded up to 64 (keeps 16-byte alignment)
    DevState st;
    int live_slot;
    // grouped launch (GROUPED kernels): 128-row tile mt of A and Y belongs
    // to expert tile_expert[mt], whose weights are W + expert * wstride (the
    // tensor map's third coordinate)
    const int* tile_expert;
    int64_t wstride;
};

// The up to 7 rows of W past its last whole group of 8 rows (rows n8 ..
// N - 1) that fall in the tile at n0: lane j < 8 takes row n8 + j, the
// segment of len bytes at koff, into dst + j * rs. Pass 0 stores the bytes
// past the last 16-byte boundary of W with plain loads and returns the bytes
// of the lane's 1-D bulk copy (from the 16-byte boundary at or below the
// segment); pass 1 issues that copy on bar. Out of line: only the last tile
// of a matrix with N % 8 != 0 runs it, and the producers' registers are few.
__device__ __noinline__ uint32_t raw_tail_rows(const uint8_t* W, int64_t N, int64_t n8, int64_t rowbytes,
                                               int64_t total_bytes, int lane, int64_t n0, int64_t koff, int64_t len,
                                               uint32_t dst, uint32_t rs, uint32_t bar, int pass) {
    const int64_t ng = n8 + lane;
    if (lane >= 8 || ng >= N || ng < n0 || ng >= n0 + BN) return 0;
    const int64_t tb16 = total_bytes & ~static_cast<int64_t>(15);
    const int64_t st = ng * rowbytes + koff;
    const int64_t s16 = st & ~static_cast<int64_t>(15);
    const int64_t e16 = min((st + len + 15) & ~static_cast<int64_t>(15), tb16);
    const uint32_t d = dst + static_cast<uint32_t>(lane) * rs;
    if (pass == 0) {
        for (int64_t q = max(e16, s16); q < st + len; ++q) sts_u8(d + static_cast<uint32_t>(q - s16), W[q]);
        return e16 > s16 ? static_cast<uint32_t>(e16 - s16) : 0u;
    }
    if (e16 > s16) bulk_g2s(d, W + s16, static_cast<uint32_t>(e16 - s16), bar);
    return 0;
}

template <int FMT, bool EXP, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap pmap) {
    constexpr bool Q6 = (FMT == FMT_Q6_K);
    constexpr int DR = Q6 ? DR_Q6K : DR_Q40;
    constexpr int RS = EXP ? kRawScale : (Q6 ? kRawQ6K : kRawQ40);
    constexpr uint32_t RW = EXP ? kPlaneTile : 0u;  // offset of the row area in a raw stage
    const SmemLayout L = smem_layout(FMT, EXP);
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t S = smem_u32(smem);
    const uint32_t BARS = S + L.bars;
    const uint32_t FLAG = S + L.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nkb = a.K / 32;  // K blocks of a row (the operands' strides)
    // this CTA's K range: blocks kbg .. kbg + nkb32 - 1 (local index kb = 0 ..)
    const int64_t kbg = static_cast<int64_t>(blockIdx.z) * a.kb_split;
    const uint32_t nkb32 = static_cast<uint32_t>(min(a.kb_split, nkb - kbg));
    const int64_t nsc = (nkb32 + 7) / 8;      // 256-column super-chunks of the range
    const int64_t sc0 = kbg / 8;              // the range's first super-chunk
    const int64_t mt = blockIdx.y, nt = blockIdx.x;
    const int64_t n0 = nt * BN;

    grid_launch_dependents();
    live_bump(a.st, a.live_slot);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full(BARS, s), 1 + kConvWarps);  // the A copy (with its bytes) and the converters
            mbar_init(bar_empty(BARS, s), 1);              // the MMA commit
        }
        for (int r = 0; r < NR; ++r) {
            mbar_init(bar_raw_full(BARS, r), 1);
            mbar_init(bar_raw_empty(BARS, r), kConvWarps);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(bar_acc_full(BARS, i), 1);
            mbar_init(bar_acc_empty(BARS, i), kEpiWarps);  // the epilogue warps
        }
        for (int i = 0; i < DR; ++i) mbar_init(bar_dv_full(BARS, i), 4);  // converters of rows 0..127
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(FLAG), "r"(0u) : "memory");
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(S + L.tslot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = lds_u32(S + L.tslot);
    // the quantized activations come from the previous kernel on the stream
    grid_dependency_wait();
    // End of a K pass, by all 896 threads (one barrier with an OR
    // reduction): another pass follows if any thread asks for one. Only the
    // converters do, at the end of the first pass of a tile that held a scale
    // beyond kScMax, so every thread makes the same number of calls. The
    // barrier is the non-aligned form, which counts threads one by one: a
    // warp whose lanes arrive apart (after lane-dependent copies) still
    // counts 32. (After an abort the second pass's waits give up at once.)
    auto next_pass = [](bool want) -> bool {
        QMM_TRACE(50, want);
        __syncwarp();
        uint32_t more;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "barrier.red.or.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(more)
            : "r"(static_cast<uint32_t>(want)), "n"(kThreads)
            : "memory");
        QMM_TRACE(51, more);
        return more != 0;
    };

    // Registers move between warpgroups (warpgroup-wide instructions): the
    // first warpgroup (producers, MMA issue, one idle warp) gives up most of
    // its share, the epilogue's two warpgroups take it.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(reg_split(FMT, EXP, GROUPED).low));
    if (warp == 0 || warp == kRawWarp) {
        // ------------------------------------------------------------ producers
        // the tile's expert (grouped launches)
        const int ex = GROUPED ? __ldg(a.tile_expert + mt) : 0;
        // raw stage of 256-column chunk scl of the range into slot r (the
        // slots cycle over the chunks of all passes)
        auto issue_raw = [&](uint32_t scl, int r) {
            const int64_t sc = sc0 + scl;  // the chunk within the row
            const uint32_t dst0 = S + L.raw + static_cast<uint32_t>(r) * L.rawslot;
            const uint32_t bar = bar_raw_full(BARS, r);
            uint32_t bytes = 0;
            // rows of whole groups of 8 through the tensor map (8 boxes),
            // the up to 7 rows past them as 1-D copies from the 16-byte
            // boundary at or below each row segment (plain loads for bytes
            // past the last 16-byte boundary of W); the plane variant takes
            // only each row's scales and d from W, and its plane tile as 16
            // boxes of 16 columns
            const int64_t koff = EXP ? sc * 210 + 192 : (Q6 ? sc * 210 : sc * 8 * 18);
            const int64_t len = EXP ? 18 : (Q6 ? 210 : min(static_cast<int64_t>(8), a.nb - sc * 8) * 18);
            const uint32_t rw0 = dst0 + RW;
            const bool boxes = n0 < a.n8;
            // the tile holds rows past W's last whole group of 8 (last tile only)
            const bool tail = a.n8 < a.N && n0 + BN > a.n8;
            if (tail)
                bytes = raw_tail_rows(GROUPED ? a.W + static_cast<int64_t>(ex) * a.wstride : a.W, a.N, a.n8,
                                      a.rowbytes, a.total_bytes, lane, n0, koff, len, rw0 + 8u * 16u * RS, RS, bar, 0);
            fence_proxy_async_smem();
            bytes = __reduce_add_sync(0xffffffffu, bytes);
            if (lane == 0)
                mbar_arrive_expect_tx(bar, bytes + (boxes ? 8u * 16u * RS : 0u) + RW);
            __syncwarp();
            if (boxes && lane < 8) {
                const int64_t xb = (lane * a.rowbytes + koff) & ~static_cast<int64_t>(15);
                if constexpr (GROUPED)
                    tma_load_3d(rw0 + lane * 16u * RS, &wmap, static_cast<int>(xb / 2), static_cast<int>(n0 / 8), ex,
                                bar);
                else
                    tma_load_2d(rw0 + lane * 16u * RS, &wmap, static_cast<int>(xb / 2), static_cast<int>(n0 / 8),
                                bar);
            }
            if (EXP && lane < 16)
                tma_load_2d(dst0 + lane * (BN * 16u), &pmap, static_cast<int>(sc * 256 + 16 * lane),
                            static_cast<int>(n0), bar);
            if (tail)
                (void)raw_tail_rows(GROUPED ? a.W + static_cast<int64_t>(ex) * a.wstride : a.W, a.N, a.n8,
                                    a.rowbytes, a.total_bytes, lane, n0, koff, len, rw0 + 8u * 16u * RS, RS, bar, 1);
        };
        if (warp == kRawWarp) {
            uint32_t r = 0, eph = 1;  // raw slot; parity of its release ((g / NR) - 1) & 1
            uint32_t g = 0;           // chunks issued, over the passes
            const uint32_t nsc32 = static_cast<uint32_t>(nsc);
            // each pass (a wait that gives up ends it), then the pass barrier
            do {
                for (uint32_t sc = 0; sc < nsc32; ++sc) {
                    QMM_TRACE(1, sc);
                    if (g >= NR && !wait_or_abort(bar_raw_empty(BARS, static_cast<int>(r)), eph, FLAG, a.st.err))
                        break;
                    issue_raw(sc, static_cast<int>(r));
                    ++g;
                    if (++r == NR) {
                        r = 0;
                        eph ^= 1;
                    }
                }
            } while (next_pass(false));
            // the copies still in flight land before the CTA ends
            for (uint32_t c = g > NR ? g - NR : 0; c < g; ++c)
                (void)wait_or_abort(bar_raw_full(BARS, static_cast<int>(c % NR)), (c / NR) & 1, FLAG, a.st.err);
        } else {
            const uint16_t* a16t = a.a16 + (mt * nkb + kbg) * (BM * 32);  // this CTA's first A tile
            uint32_t st = 0, eph = 1;  // stage; parity of its release ((q / NS) - 1) & 1
            uint32_t q = 0;            // stages, over the passes
            do {  // each pass, then the pass barrier
            for (uint32_t kb0 = 0; kb0 < nkb32; ++q, kb0 += KP) {
                // the A tiles of blocks kb0 .. (consecutive in the pre-tiled operand)
                const uint32_t nbk = nkb32 - kb0 < KP ? nkb32 - kb0 : KP;
                QMM_TRACE(2, kb0);
                if (q >= NS && !wait_or_abort(bar_empty(BARS, static_cast<int>(st)), eph, FLAG, a.st.err)) break;
                QMM_TRACE(3, kb0);
                if (lane == 0) {
                    // pull the tiles kPrefetch stages ahead into L2 first: the
                    // copy into shared memory then waits on L2, not on DRAM
                    const uint32_t pk = kb0 + kPrefetch * KP;
                    if (kb0 == 0)
                        for (uint32_t k = 0; k < pk && k < nkb32; k += KP)
                            prefetch_l2(a16t + static_cast<size_t>(k) * (BM * 32),
                                        (nkb32 - k < KP ? nkb32 - k : KP) * kATile);
                    if (pk < nkb32)
                        prefetch_l2(a16t + static_cast<size_t>(pk) * (BM * 32),
                                    (nkb32 - pk < KP ? nkb32 - pk : KP) * kATile);
                    mbar_arrive_expect_tx(bar_full(BARS, static_cast<int>(st)), nbk * kATile);
                    bulk_g2s(S + L.a + st * kAStage, a16t + static_cast<size_t>(kb0) * (BM * 32), nbk * kATile,
                             bar_full(BARS, static_cast<int>(st)));
                }
                __syncwarp();
                if (++st == NS) {
                    st = 0;
                    eph ^= 1;
                }
            }
            } while (next_pass(false));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        constexpr uint32_t idesc = idesc_f16(BM, BN);
        uint32_t st = 0, fph = 0;   // stage; parity of its fill (q / NS) & 1
        uint32_t q = 0;             // stages, over the passes
        do {  // each pass, then the pass barrier
        for (uint32_t kb0 = 0; kb0 < nkb32; ++q, kb0 += KP) {
            const uint32_t nbk = nkb32 - kb0 < KP ? nkb32 - kb0 : KP;
            QMM_TRACE(10, kb0);
            if (!wait_or_abort(bar_full(BARS, static_cast<int>(st)), fph, FLAG, a.st.err)) break;
            // stage q accumulates into buffers 2 (q % 2) + bi, free once the
            // epilogue has drained stage q - 2
            if (q >= 2 && !wait_or_abort(bar_acc_empty(BARS, static_cast<int>(q & 1)), ((q >> 1) - 1) & 1, FLAG,
                                         a.st.err))
                break;
            QMM_TRACE(12, kb0);
            tc_fence_after();
            if (lane == 0) {
                for (uint32_t bi = 0; bi < nbk; ++bi) {
                    const uint64_t ad = smem_desc(S + L.a + st * kAStage + bi * kATile);
                    const uint64_t bd = smem_desc(S + L.b + st * kBStage + bi * kBTile, kBSbo);
                    const uint32_t d = tmem + (2 * (q & 1) + bi) * BN;
                    tc_mma(d, ad, bd, idesc, 0u);
                    tc_mma(d, ad + (256 >> 4), bd + (256 >> 4), idesc, 1u);  // K columns 16..31
                }
                tc_commit(bar_acc_full(BARS, static_cast<int>(q & 1)));
                tc_commit(bar_empty(BARS, static_cast<int>(st)));
            }
            __syncwarp();
            if (++st == NS) {
                st = 0;
                fph ^= 1;
            }
            QMM_TRACE(14, kb0);
        }
        } while (next_pass(false));
    } else {
        // the idle warp keeps the pass barrier's count
        while (next_pass(false)) {
        }
    }
    } else if (warp < kEpi0) {
        if constexpr (reg_split(FMT, EXP, GROUPED).conv != 72)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(reg_split(FMT, EXP, GROUPED).conv));
        // ------------------------------------------------------------ converters
        // One stage (two K blocks) per iteration: one wait, one proxy fence and
        // one arrival. Warp cw converts the rows 8 g + cw of the tile (the plane
        // variant: g + 16 cw): lane (g = lane % 16, hh = lane / 16) the 16
        // columns 16 hh .. 16 hh + 15 of each block. In the raw stage of q6_K
        // / Q4_0 rows, a row's offset inside its slot depends only on cw, so
        // the realignment of its bytes is the same for the whole warp; plane
        // bytes need none.
        static_assert(kConvRows == 1 && KP == 2, "a converter iteration is one row and one stage of two blocks");
        static_assert((DR & (DR - 1)) == 0, "the d ring is a power of two");
        const int cw = warp - kConv0;
        const int tid = threadIdx.x - 32 * kConv0;  // rows 0..127 store d
        const int g = lane & 15, hh = lane >> 4;
        // A row's place inside a raw stage (the plane variant: its scales and
        // d), and the lead-in of its bytes there for the first 256-column
        // chunk: each further chunk moves a q6_K row by 210 = 2 (mod 16)
        // bytes and a Q4_0 row by 8 * 18 = 0 (mod 16).
        auto row_off = [&](int nn) -> uint32_t {
            const int64_t gg = n0 + nn;
            if (gg < a.n8) return RW + static_cast<uint32_t>(nn & 7) * 16u * RS + static_cast<uint32_t>(nn >> 3) * RS;
            return RW + 8u * 16u * RS + static_cast<uint32_t>(gg - a.n8) * RS;
        };
        auto lead0 = [&](int64_t gg) -> uint32_t {
            return static_cast<uint32_t>((gg * a.rowbytes + (EXP ? 192 : 0)) & 15);
        };
        const int n = EXP ? g + 16 * cw : 8 * g + cw;  // this lane's row of the tile
        const bool live = n0 + n < a.N;
        const uint32_t ro = row_off(n), l0 = live ? lead0(n0 + n) : 0u;
        const bool live_d = tid < BN && n0 + tid < a.N;  // row tid, whose d this lane stores
        const uint32_t ro_d = live_d ? row_off(tid) : 0u, l0_d = live_d ? lead0(n0 + tid) : 0u;
        uint32_t r = 0, rph = 0;   // raw slot; parity of its fill (sc / NR) & 1
        uint32_t st = 0, eph = 1;  // B stage; parity of its release ((q / NS) - 1) & 1
        uint32_t q = 0;            // stages, over the passes
        // pass 0 takes s0 of each scale; pass 1, run when some scale of the
        // tile lies beyond kScMax, takes s1 with d doubled. pf: bit 0 the
        // pass, bit 1 a scale beyond kScMax seen (one register for both).
        uint32_t pf = 0;
        for (;;) {  // each pass, then the pass barrier
        for (uint32_t kb0 = 0; kb0 < nkb32; ++q, kb0 += 2) {
            const uint32_t nbk = nkb32 - kb0 < 2 ? 1u : 2u;
            const uint32_t sc = kb0 >> 3;  // both blocks lie in this 256-column chunk
            const uint32_t j0 = kb0 & 7;
            const uint32_t raw0 = S + L.raw + r * L.rawslot;
            const uint32_t ls = Q6 ? 2u * static_cast<uint32_t>(sc0 + sc) : 0u;  // the global chunk's shift
            QMM_TRACE(20, kb0);
            if (j0 == 0 && !wait_or_abort(bar_raw_full(BARS, static_cast<int>(r)), rph, FLAG, a.st.err)) break;
            QMM_TRACE(21, kb0);
            // d of row tid (q6_K: once per super-block, Q4_0: per block), by
            // the first four converter warps (rows 0..127)
            if (tid < BN) {
                for (uint32_t bi = 0; bi < (Q6 ? (j0 == 0 ? 1u : 0u) : nbk); ++bi) {
                    // the d ring counts over the passes
                    const uint32_t di = ((pf & 1u) * (Q6 ? static_cast<uint32_t>(nsc) : nkb32) +
                                         (Q6 ? sc : kb0 + bi)) & (DR - 1);
                    float dval = 0.0f;
                    if (live_d) {
                        const uint32_t rowb = raw0 + ro_d + ((l0_d + ls) & 15u);
                        const uint32_t doff = EXP ? 16 : (Q6 ? 208 : 18 * (j0 + bi));
                        dval = half_bits_to_float(lds_u16(rowb + doff));
                        if (pf & 1u) dval += dval;  // the second pass holds s1 = (sc - s0) / 2
                    }
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(S + L.dv + (di * BN + tid) * 4), "f"(dval)
                                 : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_dv_full(BARS, static_cast<int>(di)));
                }
            }
            if (q >= NS && !wait_or_abort(bar_empty(BARS, static_cast<int>(st)), eph, FLAG, a.st.err)) break;
            QMM_TRACE(22, kb0);
            // Per row, the raw bytes of both blocks of the stage are loaded
            // first, then realigned by the row's lead (warp-uniform for rows
            // 8 g + cw), expanded and stored.
            {
                const uint32_t rb = raw0 + ro + ((l0 + ls) & 15u);
                uint32_t hv[KP][8];
                if (Q6) {
                    uint32_t c[KP][4];
                    int scv[KP];
                    if (EXP) {
#pragma unroll
                        for (int bi = 0; bi < KP; ++bi) {
                            const int e = 32 * (j0 + bi) + 16 * hh;
                            if (live && bi < nbk) {
                                lds_v4(raw0 + (e >> 4) * (BN * 16) + n * 16, c[bi]);
                                scv[bi] = lds_s8(rb + (e >> 4));
                            } else {
#pragma unroll
                                for (int w = 0; w < 4; ++w) c[bi][w] = 0x80808080u;
                                scv[bi] = 0;
                            }
                        }
#pragma unroll
                        for (int bi = 0; bi < KP; ++bi)
#pragma unroll
                            for (int w = 0; w < 4; ++w) c[bi][w] ^= 0x80808080u;
                    } else {
                        uint32_t wl[KP][8], wh[KP][8];
                        const uint32_t ab = rb & ~15u;
#pragma unroll
                        for (int bi = 0; bi < KP; ++bi) {
                            const int e = 32 * (j0 + bi) + 16 * hh;
                            if (live && bi < nbk) {
                                lds_v4(ab + (e & 127), wl[bi]);
                                lds_v4(ab + (e & 127) + 16, wl[bi] + 4);
                                lds_v4(ab + 128 + (e & 63), wh[bi]);
                                lds_v4(ab + 128 + (e & 63) + 16, wh[bi] + 4);
                                scv[bi] = lds_s8(rb + 192 + (e >> 4));
                            } else {
#pragma unroll
                                for (int w = 0; w < 8; ++w) wl[bi][w] = wh[bi][w] = 0u;
                                scv[bi] = 0;
                            }
                        }
                        uint32_t ql[KP][4], qh[KP][4];
                        pick16x4(wl[0], wl[1], wh[0], wh[1], rb & 15u, ql[0], ql[1], qh[0], qh[1]);
#pragma unroll
                        for (int bi = 0; bi < KP; ++bi) {
                            const int e = 32 * (j0 + bi) + 16 * hh;
                            const uint32_t ns = 4u * static_cast<uint32_t>(e >> 7);
                            const uint32_t hs = 2u * static_cast<uint32_t>(e >> 6);
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                c[bi][w] = ((ql[bi][w] >> ns) & 0x0F0F0F0Fu) | (((qh[bi][w] >> hs) & 0x03030303u) << 4);
                        }
                    }
#pragma unroll
                    for (int bi = 0; bi < KP; ++bi) {
                        // this pass's part s of sc; s * (v - off) exactly:
                        // (off + v) * s - off * s, one rounding
                        // (s0 = sc clamped to +-56, or to +-55 for odd sc,
                        // so that sc - s0 is even; s1 = (sc - s0) / 2)
                        const int lim = kScMax - (scv[bi] & 1);
                        const int s0 = min(max(scv[bi], -lim), lim);
                        pf |= static_cast<uint32_t>(s0 != scv[bi]) << 1;
                        const float scf = static_cast<float>((pf & 1u) ? (scv[bi] - s0) >> 1 : s0);
                        const float off = EXP ? 1152.0f : 1056.0f;
                        const uint32_t sc2 = half2_bits(scf);
                        const uint32_t bias = half2_bits(-off * scf);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            hv[bi][2 * w] = hfma2_u(half_pair_lo(c[bi][w]), sc2, bias);
                            hv[bi][2 * w + 1] = hfma2_u(half_pair_hi(c[bi][w]), sc2, bias);
                        }
                    }
                } else {
                    // Q4_0 block: nibble hh of the 16 qs bytes
                    uint32_t wq[KP][8];
#pragma unroll
                    for (int bi = 0; bi < KP; ++bi) {
                        const uint32_t qa = rb + 18 * (j0 + bi) + 2;
                        if (live && bi < nbk) {
                            lds_v4(qa & ~15u, wq[bi]);
                            lds_v4((qa & ~15u) + 16, wq[bi] + 4);
                        } else {
#pragma unroll
                            for (int w = 0; w < 8; ++w) wq[bi][w] = 0u;
                        }
                    }
                    const uint32_t ns = 4u * static_cast<uint32_t>(hh);
                    const uint32_t one = 0x3C003C00u, bias = half2_bits(-1032.0f);
#pragma unroll
                    for (int bi = 0; bi < KP; ++bi) {
                        uint32_t q[4];
                        pick16(wq[bi], (rb + 18 * (j0 + bi) + 2) & 15u, q);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const uint32_t cq = (q[w] >> ns) & 0x0F0F0F0Fu;
                            hv[bi][2 * w] = hfma2_u(half_pair_lo(cq), one, bias);
                            hv[bi][2 * w + 1] = hfma2_u(half_pair_hi(cq), one, bias);
                        }
                    }
                }
                // row n: group n / 8, row n % 8 of the group; columns 16 hh ..
                // + 15 are the K octets 2 hh and 2 hh + 1
#pragma unroll
                for (int bi = 0; bi < KP; ++bi) {
                    if (bi >= nbk) break;
                    if (!live) {
#pragma unroll
                        for (int w = 0; w < 8; ++w) hv[bi][w] = 0u;
                    }
                    const uint32_t bt = S + L.b + static_cast<uint32_t>(st) * kBStage +
                                        static_cast<uint32_t>(bi) * kBTile + (n >> 3) * kBSbo + (n & 7) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(bt + (2 * hh) * 128),
                                 "r"(hv[bi][0]), "r"(hv[bi][1]), "r"(hv[bi][2]), "r"(hv[bi][3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(bt + (2 * hh + 1) * 128),
                                 "r"(hv[bi][4]), "r"(hv[bi][5]), "r"(hv[bi][6]), "r"(hv[bi][7])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full(BARS, static_cast<int>(st)));
            QMM_TRACE(23, kb0);
            if (++st == NS) {
                st = 0;
                eph ^= 1;
            }
            if (j0 + nbk == 8 || kb0 + nbk == nkb32) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_raw_empty(BARS, static_cast<int>(r)));
                if (++r == NR) {
                    r = 0;
                    rph ^= 1;
                }
            }
        }
        if (!next_pass(pf == 2u)) break;  // first pass, a scale beyond kScMax
        pf = 1u;
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(reg_split(FMT, EXP, GROUPED).epi));
        // ------------------------------------------------------------ epilogue
        // One wait per stage of KP blocks (the MMA signals a stage once), then
        // per K block b: I_b from its accumulator buffer in two 16-column
        // tensor-memory loads and y += (I_b * D) * s_x[m][b] in registers (a
        // packed multiply and a packed FMA per two values; D is d of the
        // block's super-block for q6_K, of the block for Q4_0, read from
        // shared memory). The stage's buffers are released together.
        const int quad = warp & 3;                  // tensor-memory lanes 32*quad .. +31 (warp id mod 4)
        const int h = (warp - kEpi0) >> 2;          // columns kEpiCols*h .. of the tile
        const int64_t m = mt * BM + 32 * quad + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
        const uint32_t c0 = static_cast<uint32_t>(kEpiCols * h);
        float y[kEpiCols];  // the output
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) y[c] = 0.0f;
        float sxa[KP], sxb[KP];
        const float* xrow = a.xs + (m < a.M ? m : 0) * nkb + kbg;
        auto load_sx = [&](uint32_t k0, float (&o)[KP]) {
#pragma unroll
            for (int bi = 0; bi < KP; ++bi) {
                const uint32_t kb = k0 + bi;
                o[bi] = 0.0f;
                if (m < a.M && kb < nkb32) asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(o[bi]) : "l"(xrow + kb));
            }
        };
        bool ok = true;
        uint32_t qg = 0;     // stages, over the passes (accumulator buffers)
        uint32_t dbase = 0;  // d ring entries of the earlier passes
        for (;;) {  // each pass, then the pass barrier
        load_sx(0, sxa);
        for (uint32_t kb0 = 0; ok && kb0 < nkb32; ++qg, kb0 += KP) {
            const uint32_t nbk = nkb32 - kb0 < KP ? nkb32 - kb0 : KP;
            load_sx(kb0 + KP, sxb);
            QMM_TRACE(30, kb0);
            if (!wait_or_abort(bar_acc_full(BARS, static_cast<int>(qg & 1)), (qg >> 1) & 1, FLAG, a.st.err)) {
                ok = false;
                break;
            }
            QMM_TRACE(31, kb0);
            tc_fence_after();
            for (uint32_t bi = 0; bi < nbk; ++bi) {
                const uint32_t kb = kb0 + bi;
                // index of the d in use, counted over the passes
                const uint32_t dk = dbase + (Q6 ? kb >> 3 : kb);
                const uint32_t di = dk & (DR - 1);
                if ((!Q6 || (kb & 7) == 0) &&
                    !wait_or_abort(bar_dv_full(BARS, static_cast<int>(di)), (dk / DR) & 1, FLAG, a.st.err)) {
                    ok = false;
                    break;
                }
                const float sx = bi == 0 ? sxa[0] : sxa[1];
                const float2 s2 = make_float2(sx, sx);
                const uint32_t accb = tl + (2 * (qg & 1) + bi) * BN + c0;
                const uint32_t dv = S + L.dv + (di * BN + c0) * 4;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float v[16];
                    tc_ld16(accb + 16 * hf, v);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; c += 4) {
                        float4 d4;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(d4.x), "=f"(d4.y), "=f"(d4.z), "=f"(d4.w)
                                     : "r"(dv + 4 * (16 * hf + c)));
                        float* yy = y + 16 * hf + c;
                        const float2 t0 = ffma2(fmul2(make_float2(v[c], v[c + 1]), make_float2(d4.x, d4.y)), s2,
                                                make_float2(yy[0], yy[1]));
                        const float2 t1 = ffma2(fmul2(make_float2(v[c + 2], v[c + 3]), make_float2(d4.z, d4.w)), s2,
                                                make_float2(yy[2], yy[3]));
                        yy[0] = t0.x;
                        yy[1] = t0.y;
                        yy[2] = t1.x;
                        yy[3] = t1.y;
                    }
                }
                QMM_TRACE(32, kb);
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty(BARS, static_cast<int>(qg & 1)));
#pragma unroll
            for (int bi = 0; bi < KP; ++bi) sxa[bi] = sxb[bi];
        }
        if (!next_pass(false)) break;
        dbase += Q6 ? static_cast<uint32_t>(nsc) : nkb32;
        }
        if (ok && m < a.M) {
            const int64_t nb0 = n0 + c0;
            float* out = (a.part ? a.part + static_cast<int64_t>(blockIdx.z) * a.pstride : a.Y) + m * a.N + nb0;
            if (nb0 + kEpiCols <= a.N && (a.N & 3) == 0) {
#pragma unroll
                for (int c = 0; c < kEpiCols; c += 4)
                    *reinterpret_cast<float4*>(out + c) = make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]);
            } else {
                for (int c = 0; c < kEpiCols; ++c)
                    if (nb0 + c < a.N) out[c] = y[c];
            }
        }
    }
    QMM_TRACE(90, nkb);
    tc_fence_before();
    __syncthreads();
    QMM_TRACE(91, nkb);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- launch

using GemmKernel = void (*)(const GemmArgs, const CUtensorMap, const CUtensorMap);

static GemmKernel pick_gemm(int fmt, bool exp, bool grouped = false) {
    if (grouped) {
        if (exp) return nullptr;
        return fmt == FMT_Q6_K ? gemm_kernel<FMT_Q6_K, false, true> : gemm_kernel<FMT_Q4_0, false, true>;
    }
    if (fmt == FMT_Q6_K) return exp ? gemm_kernel<FMT_Q6_K, true, false> : gemm_kernel<FMT_Q6_K, false, false>;
    if (fmt == FMT_Q4_0 && !exp) return gemm_kernel<FMT_Q4_0, false, false>;
    return nullptr;
}

size_t gemm_a16_bytes(int64_t M, int64_t K) {
    return static_cast<size_t>((M + BM - 1) / BM * BM) * static_cast<size_t>(K) * 2;
}

// Y = the sum of the split partials, in split order (bitwise reproducible).
// Split z's partial starts at part + z * pstride, pstride a multiple of 4, so
// that the 16-byte loads of every split stay aligned (Y is 16-byte aligned).
__global__ void gemm_split_reduce_kernel(const float* __restrict__ part, float* __restrict__ Y, int64_t count,
                                         int64_t pstride, int splits, DevState st) {
    grid_dependency_wait();  // the GEMM's partials
    grid_launch_dependents();
    live_bump(st, 20);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < count; i += stride) {
        if (i + 4 <= count) {
            float4 acc = *reinterpret_cast<const float4*>(part + i);
            for (int z = 1; z < splits; ++z) {
                const float4 v = *reinterpret_cast<const float4*>(part + z * pstride + i);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4*>(Y + i) = acc;
        } else {
            for (int64_t j = i; j < count; ++j) {
                float acc = part[j];
                for (int z = 1; z < splits; ++z) acc += part[z * pstride + j];
                Y[j] = acc;
            }
        }
    }
}

namespace {

int sm_count() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev] = n;
    return n;
}

// K blocks per split: a grid of fewer tiles than SMs splits K so that tiles
// x splits fills the SMs, keeping at least 4 super-chunks (32 blocks) per
// split; a multiple of 8 blocks, so that splits start on super-chunks.
int64_t gemm_kb_split(int64_t M, int64_t N, int64_t K) {
    const int64_t nkb = K / 32;
    const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
    int64_t S = sm_count() / (tiles > 0 ? tiles : 1);
    if (S > nkb / 32) S = nkb / 32;
    if (S < 2) return nkb;
    const int64_t per = (nkb + S - 1) / S;
    return (per + 7) / 8 * 8;
}

}  // namespace

int gemm_splits(int64_t M, int64_t N, int64_t K) {
    const int64_t nkb = K / 32;
    const int64_t kbs = gemm_kb_split(M, N, K);
    return static_cast<int>((nkb + kbs - 1) / kbs);
}

namespace {
int64_t part_stride(int64_t M, int64_t N) { return (M * N + 63) / 64 * 64; }
}  // namespace

size_t gemm_part_bytes(int64_t M, int64_t N, int64_t K) {
    const int S = gemm_splits(M, N, K);
    return S > 1 ? static_cast<size_t>(S) * static_cast<size_t>(part_stride(M, N)) * 4 : 0;
}

cudaError_t gemm_launch(int fmt, bool exp, const uint8_t* W, const int8_t* plane,
                        const uint16_t* a16, const float* xs, float* Y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s, DevState st, int live_slot, float* part) {
    GemmKernel k = pick_gemm(fmt, exp);
    if (!k) return cudaErrorInvalidValue;
    const SmemLayout L = smem_layout(fmt, exp);
    static std::mutex mu;
    static std::map<std::pair<int, GemmKernel>, bool> ready;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!ready[{dev, k}]) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(L.total));
            if (e != cudaSuccess) return e;
            ready[{dev, k}] = true;
        }
    }
    GemmArgs a{};
    a.W = W;
    a.plane = plane;
    a.a16 = a16;
    a.xs = xs;
    a.Y = Y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.nb = K / (fmt == FMT_Q6_K ? 256 : 32);
    a.total_bytes = N * a.nb * (fmt == FMT_Q6_K ? 210 : 18);
    a.rowbytes = a.nb * (fmt == FMT_Q6_K ? 210 : 18);
    a.n8 = N / 8 * 8;
    a.st = st;
    a.live_slot = live_slot;
    a.kb_split = gemm_kb_split(M, N, K);
    const int splits = gemm_splits(M, N, K);
    if (splits > 1 && !part) return cudaErrorInvalidValue;
    a.part = splits > 1 ? part : nullptr;
    a.pstride = part_stride(M, N);
    if (a.part && (reinterpret_cast<uintptr_t>(part) & 15u)) return cudaErrorMisalignedAddress;
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM),
                    static_cast<unsigned>(splits));
    // q6_K / Q4_0 rows: W as [N / 8][8 * rowbytes] bytes of 16-bit elements
    // (the pitch of 8 rows is a multiple of 16 bytes for both formats); a box
    // is one row slot wide and 16 groups of 8 rows high
    // (the plane variant: 48-byte boxes of each row's scales and d); the
    // plane as [N][K] bytes, a box 16 columns wide and 128 rows high
    CUtensorMap wmap, pmap;
    memset(&wmap, 0, sizeof wmap);
    memset(&pmap, 0, sizeof pmap);
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    if (exp) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
        const cuuint32_t box[2] = {16u, static_cast<cuuint32_t>(BN)};
        const cuuint32_t es[2] = {1u, 1u};
        if (enc(&pmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(plane), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (a.n8 > 0) {
        const int rs = exp ? kRawScale : (fmt == FMT_Q6_K ? kRawQ6K : kRawQ40);
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(4 * a.rowbytes), static_cast<cuuint64_t>(a.n8 / 8)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(8 * a.rowbytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(rs / 2), 16u};
        const cuuint32_t es[2] = {1u, 1u};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t*>(W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    e = launch_pdl(k, grid, dim3(kThreads), L.total, s, a, wmap, pmap);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    const int64_t count = M * N;
    int64_t blocks = (count / 4 + 255) / 256;
    if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
    if (blocks < 1) blocks = 1;
    e = launch_pdl(gemm_split_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                   static_cast<const float*>(part), Y, count, a.pstride, splits, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t gemm_grouped_launch(int fmt, const uint8_t* W, int64_t wstride, int n_experts, const int* tile_expert,
                                const uint16_t* a16, const float* xs, float* Y, int64_t M, int64_t N, int64_t K,
                                cudaStream_t s, DevState st, int live_slot) {
    GemmKernel k = pick_gemm(fmt, false, true);
    if (!k) return cudaErrorInvalidValue;
    if (M % BM || wstride % 16 || n_experts < 1) return cudaErrorInvalidValue;
    const SmemLayout L = smem_layout(fmt, false);
    static std::mutex mu;
    static std::map<std::pair<int, GemmKernel>, bool> ready;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!ready[{dev, k}]) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
            if (e != cudaSuccess) return e;
            ready[{dev, k}] = true;
        }
    }
    GemmArgs a{};
    a.W = W;
    a.a16 = a16;
    a.xs = xs;
    a.Y = Y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.nb = K / (fmt == FMT_Q6_K ? 256 : 32);
    a.total_bytes = N * a.nb * (fmt == FMT_Q6_K ? 210 : 18);
    a.rowbytes = a.nb * (fmt == FMT_Q6_K ? 210 : 18);
    a.n8 = N / 8 * 8;
    a.st = st;
    a.live_slot = live_slot;
    a.kb_split = K / 32;  // one split: the tiles of all experts fill the SMs
    a.part = nullptr;
    a.pstride = part_stride(M, N);
    a.tile_expert = tile_expert;
    a.wstride = wstride;
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>(M / BM), 1u);
    // W of every expert as [E][N / 8][8 * rowbytes] 16-bit elements, experts
    // wstride bytes apart; a box one row slot wide, 16 groups of 8 rows high
    CUtensorMap wmap, pmap;
    memset(&wmap, 0, sizeof wmap);
    memset(&pmap, 0, sizeof pmap);
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    if (a.n8 > 0) {
        const int rs = fmt == FMT_Q6_K ? kRawQ6K : kRawQ40;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(4 * a.rowbytes), static_cast<cuuint64_t>(a.n8 / 8),
                                    static_cast<cuuint64_t>(n_experts)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(8 * a.rowbytes), static_cast<cuuint64_t>(wstride)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(rs / 2), 16u, 1u};
        const cuuint32_t es[3] = {1u, 1u, 1u};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t*>(W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    e = launch_pdl(k, grid, dim3(kThreads), L.total, s, a, wmap, pmap);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace qmm
