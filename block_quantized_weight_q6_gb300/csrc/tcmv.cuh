// tcmv.cuh -- fused dequantize + matvec for 1..16 activation rows on the
// sm_103a tensor cores; included by one translation unit per weight format.
//
//   y[b][n] = sum_g s[n][g] * P[b][n][g],   P[b][n][g] = sum_{k in g} c[n][k] * x[b][k]
//
// c is the weight's exact small-integer code and g its scale group:
//   q6_K  c = q - 32, groups of 16, s = d * scales[g]
//   Q4_0  c = q - 8,  groups of 32, s = d
//   Q8_0  c = q,      groups of 32, s = d
// Every code is an exact bf16 value, and so is a bf16 activation; an fp32
// activation is split exactly into three bf16 terms (hi + mid + lo) that
// take three MMA columns. Every product is therefore exact and P is an fp32
// sum of exact products, formed by tcgen05.mma (kind::f16, bf16 operands,
// fp32 accumulator in tensor memory):
//   A  128 weight rows x 16 K in tensor memory, written row-per-thread by the
//      decoding warps with tcgen05.st (lane = row, column c = K pair 2c, 2c+1);
//   B  16 / 32 / 48 activation columns x 16 K in shared memory: the
//      activation tile prepared once per call, one bulk copy per stage;
//   D  one 128 x N accumulator per scale group in tensor memory, drained by
//      the same decoding threads with tcgen05.ld, which apply s and sum.
// In q8 mode the activations are the per-32 int8 codes (exact in bf16), P is
// the exact integer partial, and y = sum s_x[b][blk] * s[n][g] * P.
//
// Why the tensor cores for a matvec (quantprobe "LAWS.md", Law 4 amendments
// L-15 / L-16: the unpack instruction cost, not the bit width, sets decode
// speed): on the CUDA cores every weight costs its unpack plus one FMA per
// activation row, and at 8 rows the FP32 pipe alone cannot keep up with HBM.
// Here the unpack ends at an exact bf16 code (one byte-permute and one packed
// bf16 FMA per two weights) and the activation rows ride in MMA columns.
//
// CTA (768 threads, one per SM, persistent over work items = 128-row tile x
// a range of 256-wide K stages), warps by role:
//   0-15   decoders: two sets of 8 warps take alternate stages; in a set,
//          warps w and w + 4 cover the same tensor-memory lanes and split the
//          quads of each half stage (row = tc_lane_row(32 * (warp % 4) + lane))
//   16-19  drainers: load the accumulators, apply the scales, sum, store
//   20     weight producer: per stage, 8 tensor-map copies of the tile's raw
//          blocks (W seen as rows of 8 weight rows: any row pitch becomes a
//          16-byte multiple, and one copy brings row j of 16 such groups),
//          1-D bulk copies for the rows past the last whole group of 8
//   21-22  MMA issue, one thread per decode set; warp 21 owns the tensor memory
//   23     activation producer: builds each stage's B operand (float mode) or
//          copies the prepared one (q8 mode)
// Rings, each slot with a full / empty mbarrier pair, every wait bounded in
// time: raw weight stages (producer -> decoders), activation stages
// (producer -> MMA), group scales (decoders -> drainers), A half stages per
// decode set (decoders -> MMA), D windows (MMA -> drainers). A raw stage is
// free again as soon as it has been decoded.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "tc.cuh"

namespace qmm {

constexpr int kTcStageK = 256;      // K elements per stage
constexpr uint32_t kTcSmemCap = 226u * 1024;  // dynamic shared memory per CTA at most

// Per format: block bytes, blocks per stage, row slot stride in a raw stage,
// K width of a scale group, quads per stage, A columns per group.
template <int FMT>
struct TcF;
template <>
struct TcF<FMT_Q6_K> {
    // one 210-byte super-block per row per stage; a quad is the 4 groups
    // q, q+4, q+8, q+12 that share one run of 16 qh bytes
    static constexpr int BB = 210, BPS = 1, RS = 240, GK = 16, QPS = 4, GA = 8;
};
template <>
struct TcF<FMT_Q4_0> {
    static constexpr int BB = 18, BPS = 8, RS = 176, GK = 32, QPS = 2, GA = 16;
};
template <>
struct TcF<FMT_Q8_0> {
    static constexpr int BB = 34, BPS = 8, RS = 304, GK = 32, QPS = 2, GA = 16;
};

// Row slot strides are 16 * odd (conflict-free 16-byte loads across rows) and
// hold the longest copy (payload + 2 * 14 bytes of 16-byte rounding) plus the
// one-word over-read of the unaligned loads.
static_assert(TcF<FMT_Q6_K>::RS % 32 == 16 && TcF<FMT_Q4_0>::RS % 32 == 16 &&
                  TcF<FMT_Q8_0>::RS % 32 == 16,
              "row slot stride");
static_assert(210 + 28 <= 240 && 8 * 18 + 28 <= 176 && 8 * 34 + 28 <= 304, "row slot size");

template <int NB, int S>
struct TcCols {
    static constexpr int NC = NB * S;  // activation columns in use
    // MMA N: wider than a group needs when a group takes 4 to 8 columns (32
    // for 4-5, 64 for 6-8), so that a D window collects several groups and a
    // stage needs few windows (fewer drains); else the smallest of 16, 32, 48
    // that holds a group
    static constexpr int NCOL = (NC >= 6 && NC <= 8) ? 64
                              : (NC >= 4 && NC <= 5) ? 32
                              : (NC <= 16 ? 16 : (NC <= 32 ? 32 : 48));
};

template <int FMT, int NB, int S>
struct TcLayout {
    using F = TcF<FMT>;
    static constexpr int NCOL = TcCols<NB, S>::NCOL;
    // raw slot: 8 boxes (row j of every group of 8 rows, 16 groups per tile),
    // rows one slot RS apart, then a tail area for the up to 7 rows past the
    // last whole group of 8; tensor-map destinations are 128-byte aligned
    static constexpr uint32_t BOXP = 16u * F::RS;
    static_assert(BOXP % 128 == 0 && (8u * F::RS) % 128 == 0, "box alignment");
    static constexpr uint32_t TAIL = 8 * BOXP;
    static constexpr uint32_t RAW = TAIL + 8u * F::RS;
    // activation slot: the stage's 16 K16-step B operands
    static constexpr uint32_t XT = static_cast<uint32_t>(NCOL) * kTcStageK * 2;
    static constexpr int QA = 4 * F::GA;                       // A columns per quad
    static constexpr int SA = F::QPS * QA;                     // A columns per stage (128)
    static constexpr int GPS = 4 * F::QPS;                     // scale groups per stage
    // scale slot: the stage's group scales, [group][tensor-memory lane] fp32
    static constexpr uint32_t SCB = static_cast<uint32_t>(GPS) * 128 * 4;
    // D windows: NCOL columns (one MMA's N), aligned. A window collects the
    // partial sums of G = NCOL / NC consecutive groups (issue order i = 4Q + g):
    // group i's activations fill rows (i % G) * NC .. + NC - 1 of its B
    // operand and every other row is zero, so each group's MMAs add only into
    // its own NC columns; the first MMA into a window starts it from zero.
    static constexpr int NC = NB * S;                          // columns per group
    static constexpr int G = NCOL / NC;                        // groups per window
    static constexpr int W = (GPS + G - 1) / G;                // windows per stage
    // A half stages (SA / 2 columns) per decode set: three when a stage needs
    // at most two windows (the MMAs of a half then have a further half stage
    // of decoding to finish in), else two
    static constexpr int NAH = (NCOL == 16 && W <= 2) ? 3 : 2;
    static constexpr uint32_t DCOL0 = 2 * NAH * (SA / 2);
    static constexpr int NW0 = static_cast<int>((512 - DCOL0) / NCOL);
    static constexpr int NW = NW0 > 16 ? 16 : NW0;             // windows in flight
    // each MMA issuer (decode set) has its own NWS windows, so a window is
    // reused only after the drain of that issuer's previous use of it, and
    // every wait targets the latest phase of its barrier
    static constexpr int NWS = NW / 2;
    static_assert(G >= 1 && NWS >= 1, "tensor memory");
    static constexpr uint32_t TNEED = DCOL0 + NW * NCOL;
    static_assert(TNEED <= 512, "tensor memory");
    // rings: raw (producer -> decoders), activations (producer -> MMA),
    // scales (decoders -> drainers)
    static constexpr int NX = NCOL == 16 ? 4 : 2;
    static constexpr int NSC = 3;
    static constexpr int NR0 =
        static_cast<int>((kTcSmemCap - NX * XT - NSC * SCB - 1024) / RAW);
    static constexpr int NR = NR0 > 6 ? 6 : NR0;
    static_assert(NR >= 3, "raw stages");
    static constexpr uint32_t XOFF = NR * RAW;
    static constexpr uint32_t SOFF = XOFF + NX * XT;
    static constexpr uint32_t BARS = SOFF + NSC * SCB;
    // barriers: r_full[NR], r_empty[NR], x_full[NX], x_empty[NX], s_full[NSC],
    // s_empty[NSC], a_full[2][NAH], a_empty[2][NAH] ([decode set][half slot]),
    // d_full[NW], d_empty[NW], final
    static constexpr uint32_t NBARS = 2 * NR + 2 * NX + 2 * NSC + 4 * NAH + 2 * NW + 1;
    static constexpr uint32_t TSLOT = BARS + 8 * NBARS;
    static constexpr uint32_t ABORT = TSLOT + 4;
    static constexpr uint32_t USED = (ABORT + 4 + 127) / 128 * 128;
    // one CTA per SM: it owns all 512 tensor-memory columns, and the
    // shared-memory request keeps a second CTA off the SM
    static constexpr uint32_t SMEM = USED > 120u * 1024 ? USED : 120u * 1024;
    static_assert(SMEM <= kTcSmemCap, "shared memory");
};

// ------------------------------------------------------------ trace
// Diagnostic builds define QMM_TCMV_TRACE and point g_tcmv_trace at a device
// buffer: CTA 0 records %globaltimer at the pipeline events of its first 64
// stages, so the stage timeline can be read from the host. Product builds
// compile it out.
#ifdef QMM_TCMV_TRACE
__device__ unsigned long long* g_tcmv_trace;
#define TCMV_TRACE(ev, i)                                                                \
    do {                                                                                 \
        if (blockIdx.x == 0 && g_tcmv_trace && (i) < 64) g_tcmv_trace[(ev) * 64 + (i)] = \
            globaltimer_ns();                                                            \
    } while (0)
#else
#define TCMV_TRACE(ev, i) \
    do {                  \
    } while (0)
#endif

// ------------------------------------------------------------ bounded waits
// A waiting thread sleeps inside try_wait (up to the hint, waking when the
// phase completes) instead of spinning: the decoding warps share the issue
// slots with every waiting role.
constexpr uint32_t kTcSleepNs = 20000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kTcSleepNs)
        : "memory");
    return ok != 0;
}

// Warp-collective wait that also gives up once another role of the CTA gave
// up; every lane leaves with the same answer (the tensor-memory operations
// that follow are .sync.aligned).
__device__ __forceinline__ bool tcmv_wait_warp(uint32_t bar, uint32_t parity, uint32_t flag,
                                               unsigned int* err,
                                               unsigned long long limit_ns = kWaitLimitNs) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity))) return true;
        if ((it & 3u) == 0) {
            int give_up = lds_u32(flag) != 0 ? 1 : 0;
            if (!give_up && globaltimer_ns() - t0 > limit_ns) give_up = 2;
            give_up = __shfl_sync(0xffffffffu, give_up, 0);
            if (give_up) {
                if (give_up == 2 && (threadIdx.x & 31) == 0) {
                    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(flag), "r"(1u) : "memory");
                    atomicOr(err, DERR_GEMV_TIMEOUT);
                }
                __syncwarp();
                return false;
            }
        }
    }
}

// The same for a single thread.
__device__ __forceinline__ bool tcmv_wait_one(uint32_t bar, uint32_t parity, uint32_t flag,
                                              unsigned int* err) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if ((it & 3u) == 0) {
            if (lds_u32(flag) != 0) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(flag), "r"(1u) : "memory");
                atomicOr(err, DERR_GEMV_TIMEOUT);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------ codes -> bf16
// Code bytes below 128 -> bf16 pairs (128 + byte) of bytes (0, 1) / (2, 3).
__device__ __forceinline__ uint32_t bf_pair_lo(uint32_t c) { return __byte_perm(c, 0x43434343u, 0x4140); }
__device__ __forceinline__ uint32_t bf_pair_hi(uint32_t c) { return __byte_perm(c, 0x43434343u, 0x4342); }

// v + c on bf16 pairs, rounded once (exact here: the results are small integers)
__device__ __forceinline__ uint32_t bf_add(uint32_t v, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(0x3F803F80u), "r"(c));
    return d;
}

constexpr uint32_t kBfNeg160 = 0xC320C320u;  // bf16 pair (-160, -160): (128 + q) - 160 = q - 32
constexpr uint32_t kBfNeg136 = 0xC308C308u;  // bf16 pair (-136, -136): (128 + q) - 136 = q - 8

// signed code bytes (Q8_0) -> two bf16 pairs, through exact fp32 values
__device__ __forceinline__ void q8_bf_pairs(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = w ^ 0x80808080u;  // q + 128, as unsigned bytes
    const float2 neg = make_float2(-(8388608.0f + 128.0f), -(8388608.0f + 128.0f));
    const float2 f01 = fadd2(make_float2(byte_as_magic_float<0>(u), byte_as_magic_float<1>(u)), neg);
    const float2 f23 = fadd2(make_float2(byte_as_magic_float<2>(u), byte_as_magic_float<3>(u)), neg);
    // |q| <= 127 has at most 7 significant bits: the upper half is the bf16
    p01 = __byte_perm(__float_as_uint(f01.x), __float_as_uint(f01.y), 0x7632);
    p23 = __byte_perm(__float_as_uint(f23.x), __float_as_uint(f23.y), 0x7632);
}

// K offset (within the 256-element stage) of group g of quad Q
template <int FMT>
__host__ __device__ constexpr int tc_group_k(int Q, int g) {
    return FMT == FMT_Q6_K ? 16 * Q + 64 * g : 32 * (4 * Q + g);
}

// x-tile scale block (32 wide) of group g of quad Q, relative to the stage
template <int FMT>
__device__ __forceinline__ int tc_group_xblk(int Q, int g) {
    return tc_group_k<FMT>(Q, g) >> 5;
}

// ------------------------------------------------------------ decode a stage
// Writes the A operand of every group of this thread's row in the stage into
// tensor-memory columns from `acol` (lane = this row): quad Q at acol + Q * QA,
// group g of the quad GA columns further per g. All shared-memory loads of
// the stage are issued before any arithmetic, and one wait covers all stores.
// part P of half H of the stage: q6_K quad 2H + P; Q4_0 / Q8_0 blocks
// 4H + 2P and 4H + 2P + 1
template <int FMT, int H, int P>
__device__ __forceinline__ void tc_decode_stage(uint32_t rowp, uint32_t acol) {
    using F = TcF<FMT>;
    constexpr int QA = 4 * F::GA;
    if constexpr (FMT == FMT_Q6_K) {
        uint32_t qh[4][4], qa[4][4], qb[4][4];
#pragma unroll
        for (int Q = 2 * H + P; Q < 2 * H + P + 1; ++Q) {
            lds_words_unaligned<4>(rowp + 128 + 16 * Q, qh[Q]);
            lds_words_unaligned<4>(rowp + 16 * Q, qa[Q]);
            lds_words_unaligned<4>(rowp + 64 + 16 * Q, qb[Q]);
        }
#pragma unroll
        for (int Q = 2 * H + P; Q < 2 * H + P + 1; ++Q) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                // group j = Q + 4g: ql run (j & 7), nibble j >> 3, qh field j >> 2 = g
                uint32_t A[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t base = (g & 1) ? qb[Q][w] : qa[Q][w];
                    const uint32_t nib = (g < 2) ? base : (base >> 4);
                    uint32_t h;
                    if (g == 0) h = (qh[Q][w] & 0x03030303u) << 4;
                    else if (g == 1) h = (qh[Q][w] & 0x0C0C0C0Cu) << 2;
                    else if (g == 2) h = qh[Q][w] & 0x30303030u;
                    else h = (qh[Q][w] >> 2) & 0x30303030u;
                    const uint32_t c = (nib & 0x0F0F0F0Fu) | h;
                    A[2 * w] = bf_add(bf_pair_lo(c), kBfNeg160);
                    A[2 * w + 1] = bf_add(bf_pair_hi(c), kBfNeg160);
                }
                tc::st8(acol + QA * Q + F::GA * g, A);
            }
        }
    } else if constexpr (FMT == FMT_Q4_0) {
        uint32_t qs[8][4];
#pragma unroll
        for (int i = 4 * H + 2 * P; i < 4 * H + 2 * P + 2; ++i) lds_words_unaligned<4>(rowp + F::BB * i + 2, qs[i]);
#pragma unroll
        for (int i = 4 * H + 2 * P; i < 4 * H + 2 * P + 2; ++i) {
            uint32_t A[16];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t lo = qs[i][w] & 0x0F0F0F0Fu;         // elements 4w..4w+3
                const uint32_t hi = (qs[i][w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w..
                A[2 * w] = bf_add(bf_pair_lo(lo), kBfNeg136);
                A[2 * w + 1] = bf_add(bf_pair_hi(lo), kBfNeg136);
                A[8 + 2 * w] = bf_add(bf_pair_lo(hi), kBfNeg136);
                A[8 + 2 * w + 1] = bf_add(bf_pair_hi(hi), kBfNeg136);
            }
            tc::st16(acol + QA * (i >> 2) + F::GA * (i & 3), A);
        }
    } else {
#pragma unroll
        for (int i = 4 * H + 2 * P; i < 4 * H + 2 * P + 2; ++i) {
            uint32_t qs[8];
            lds_words_unaligned<8>(rowp + F::BB * i + 2, qs);
            uint32_t A[16];
#pragma unroll
            for (int w = 0; w < 8; ++w) q8_bf_pairs(qs[w], A[2 * w], A[2 * w + 1]);
            tc::st16(acol + QA * (i >> 2) + F::GA * (i & 3), A);
        }
    }
}

// ------------------------------------------------------------ aligned decode
// When the row pitch is a multiple of 16 bytes every row of a stage has the
// same lead, so the decode is specialized on it: 16-byte shared loads from
// the 16-byte aligned row slot, and byte realignment by compile-time shifts.

__device__ __forceinline__ void lds128(uint32_t a, uint32_t* w) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(a));
}

// the 16 bytes at slot + OFF (OFF even, known at compile time) as 4 words
template <int OFF>
__device__ __forceinline__ void tc_run16(uint32_t slot, uint32_t (&o)[4]) {
    constexpr int A = OFF & ~15, Q = (OFF & 15) >> 2, SH = (OFF & 3) * 8;
    uint32_t w[8];
    lds128(slot + A, w);
    if constexpr (Q > 0 || SH > 0) lds128(slot + A + 16, w + 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = SH ? __funnelshift_r(w[Q + k], w[Q + k + 1], SH) : w[Q + k];
}

// The 16 bytes at slot + off + 4 * QW + sh / 8 (off a multiple of 16, sh 0 or
// 16) as 4 words: two 16-byte loads and a funnel shift per word.
template <int QW>
__device__ __forceinline__ void tc_run16_q(uint32_t addr, uint32_t sh, uint32_t (&o)[4]) {
    uint32_t w[8];
    lds128(addr, w);
    lds128(addr + 16, w + 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(w[QW + k], w[QW + k + 1], sh);
}

// q6_K: quad Q (runtime) of a super-block whose bytes start at slot + 4 * QW +
// sh / 8; one body per word offset QW keeps the code small
template <int QW>
__device__ __forceinline__ void tc_q6k_quad_q(uint32_t slot, int Q, uint32_t sh, uint32_t acol) {
    using F = TcF<FMT_Q6_K>;
    uint32_t qh[4], qa[4], qb[4];
    tc_run16_q<QW>(slot + 128 + 16 * Q, sh, qh);
    tc_run16_q<QW>(slot + 16 * Q, sh, qa);
    tc_run16_q<QW>(slot + 64 + 16 * Q, sh, qb);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t A[8];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t base = (g & 1) ? qb[w] : qa[w];
            const uint32_t nib = (g < 2) ? base : (base >> 4);
            uint32_t h;
            if (g == 0) h = (qh[w] & 0x03030303u) << 4;
            else if (g == 1) h = (qh[w] & 0x0C0C0C0Cu) << 2;
            else if (g == 2) h = qh[w] & 0x30303030u;
            else h = (qh[w] >> 2) & 0x30303030u;
            const uint32_t c = (nib & 0x0F0F0F0Fu) | h;
            A[2 * w] = bf_add(bf_pair_lo(c), kBfNeg160);
            A[2 * w + 1] = bf_add(bf_pair_hi(c), kBfNeg160);
        }
        tc::st8(acol + 4 * F::GA * Q + F::GA * g, A);
    }
}

// Q4_0 / Q8_0: block I of the stage, bytes from slot + LEAD + BB * I
template <int FMT, int LEAD, int I>
__device__ __forceinline__ void tc_q32_block_aligned(uint32_t slot, uint32_t acol) {
    using F = TcF<FMT>;
    constexpr int OFF = LEAD + F::BB * I + 2;
    uint32_t A[16];
    if constexpr (FMT == FMT_Q4_0) {
        uint32_t qs[4];
        tc_run16<OFF>(slot, qs);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t lo = qs[w] & 0x0F0F0F0Fu;
            const uint32_t hi = (qs[w] >> 4) & 0x0F0F0F0Fu;
            A[2 * w] = bf_add(bf_pair_lo(lo), kBfNeg136);
            A[2 * w + 1] = bf_add(bf_pair_hi(lo), kBfNeg136);
            A[8 + 2 * w] = bf_add(bf_pair_lo(hi), kBfNeg136);
            A[8 + 2 * w + 1] = bf_add(bf_pair_hi(hi), kBfNeg136);
        }
    } else {
        uint32_t q0[4], q1[4];
        tc_run16<OFF>(slot, q0);
        tc_run16<OFF + 16>(slot, q1);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            q8_bf_pairs(q0[w], A[2 * w], A[2 * w + 1]);
            q8_bf_pairs(q1[w], A[8 + 2 * w], A[8 + 2 * w + 1]);
        }
    }
    tc::st16(acol + 4 * F::GA * (I >> 2) + F::GA * (I & 3), A);
}

// The general per-row realignment, for row pitches that are not multiples of
// 16 bytes (kept out of line: the common case never runs it).
template <int FMT>
__device__ __noinline__ void tc_decode_half_general(uint32_t rowp, uint32_t acol, int h, int p) {
    if (h == 0) {
        if (p == 0) tc_decode_stage<FMT, 0, 0>(rowp, acol);
        else tc_decode_stage<FMT, 0, 1>(rowp, acol);
    } else {
        if (p == 0) tc_decode_stage<FMT, 1, 0>(rowp, acol);
        else tc_decode_stage<FMT, 1, 1>(rowp, acol);
    }
}

// Decode of part p of half h of a stage (q6_K quad 2h + p; Q4_0 / Q8_0
// blocks 4h + 2p, 4h + 2p + 1): the two 4-warp parts of a decode set share
// each half stage. When every row has the same lead (row pitch a multiple of
// 16 bytes) the loads are 16-byte loads from the aligned slot: q6_K by word
// offset of the lead (warp-uniform branch), Q4_0 / Q8_0 only at lead 0 (their
// stages are 144 / 272 bytes, so every stage starts on a 16-byte boundary).
template <int FMT>
__device__ __forceinline__ void tc_decode_half(uint32_t slot, uint32_t lead, bool uniform,
                                               uint32_t acol, int h, int p) {
    if (uniform) {
        if constexpr (FMT == FMT_Q6_K) {
            const uint32_t sh = (lead & 3u) * 8u;
            const int Q = 2 * h + p;
            switch (lead >> 2) {
                case 0: tc_q6k_quad_q<0>(slot, Q, sh, acol); break;
                case 1: tc_q6k_quad_q<1>(slot, Q, sh, acol); break;
                case 2: tc_q6k_quad_q<2>(slot, Q, sh, acol); break;
                default: tc_q6k_quad_q<3>(slot, Q, sh, acol); break;
            }
            return;
        } else {
            if (lead == 0) {
                switch (2 * h + p) {
                    case 0:
                        tc_q32_block_aligned<FMT, 0, 0>(slot, acol);
                        tc_q32_block_aligned<FMT, 0, 1>(slot, acol);
                        break;
                    case 1:
                        tc_q32_block_aligned<FMT, 0, 2>(slot, acol);
                        tc_q32_block_aligned<FMT, 0, 3>(slot, acol);
                        break;
                    case 2:
                        tc_q32_block_aligned<FMT, 0, 4>(slot, acol);
                        tc_q32_block_aligned<FMT, 0, 5>(slot, acol);
                        break;
                    default:
                        tc_q32_block_aligned<FMT, 0, 6>(slot, acol);
                        tc_q32_block_aligned<FMT, 0, 7>(slot, acol);
                        break;
                }
                return;
            }
        }
    }
    tc_decode_half_general<FMT>(slot + lead, acol, h, p);
}

// The scale of every group of this thread's row in the stage (issue order),
// stored into the scale slot at [group][lane m]. Blocks past the end of the
// row (last stage of a ragged K) hold stale bytes; their activations are zero
// and their scale is 0.
template <int FMT>
__device__ __forceinline__ void tc_store_scales(uint32_t rowp, int nblk, uint32_t sslot, int m, int p) {
    using F = TcF<FMT>;
    if constexpr (FMT == FMT_Q6_K) {
        // part p: the groups of quads p and p + 2 (issue order i = 4Q + g)
        const float d = half_bits_to_float(lds_u16(rowp + 208));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = 4 * (p + 2 * (u >> 2)) + (u & 3);
            const int j = (i >> 2) + 4 * (i & 3);  // the group's index in the super-block
            const float v = d * static_cast<float>(lds_s8(rowp + 192 + j));
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sslot + (i * 128 + m) * 4), "f"(v) : "memory");
        }
        (void)nblk;
    } else {
        // part p: blocks 2p, 2p + 1, 4 + 2p, 5 + 2p
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = 2 * p + (u & 1) + 4 * (u >> 1);
            const float d = half_bits_to_float(lds_u16(rowp + F::BB * i));
            const float v = i < nblk ? d : 0.0f;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sslot + (i * 128 + m) * 4), "f"(v) : "memory");
        }
    }
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// ------------------------------------------------------------ drain a window
// Loads the window (this thread's row) and adds s_i * (activation scale) * P
// to acc[b] for every group i of the window and every activation row b.
template <int NCOL>
__device__ __forceinline__ void tc_ld_window(uint32_t taddr, uint32_t (&v)[NCOL]) {
    if constexpr (NCOL == 64) {
        tc::ld<32>(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tc::ld<32>(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    } else if constexpr (NCOL == 48) {
        tc::ld<32>(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tc::ld<16>(taddr + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
    } else {
        tc::ld<NCOL>(taddr, v);
    }
}

template <int FMT, int NB, int S, bool Q8>
__device__ __forceinline__ void tc_drain_window(uint32_t dcol, uint32_t sslot, int m, int w,
                                                int64_t xblk0, const TcmvArgs& a, float (&acc)[NB]) {
    using L = TcLayout<FMT, NB, S>;
    constexpr int NCOL = L::NCOL, NC = L::NC, G = L::G;
    uint32_t v[NCOL];
    tc_ld_window<NCOL>(dcol, v);
    float sg[G];
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const int i = w * G + u;
        sg[u] = i < L::GPS ? lds_f32(sslot + (i * 128 + m) * 4) : 0.0f;
    }
    tc::wait_ld();
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const int i = w * G + u;
        if (i >= L::GPS) break;
        float sc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) sc[b] = sg[u];
        if constexpr (Q8) {
            // activation scales of the group's 32-block, stored [block][NB]
            const float* xs = a.xs + (xblk0 + (tc_group_k<FMT>(i >> 2, i & 3) >> 5)) * NB;
            if constexpr (NB >= 4) {
#pragma unroll
                for (int b = 0; b < NB; b += 4) {
                    const float4 f = __ldg(reinterpret_cast<const float4*>(xs + b));
                    sc[b] *= f.x;
                    sc[b + 1] *= f.y;
                    sc[b + 2] *= f.z;
                    sc[b + 3] *= f.w;
                }
            } else {
#pragma unroll
                for (int b = 0; b < NB; ++b) sc[b] *= __ldg(xs + b);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int c = u * NC + b * S;
            float p;
            if constexpr (S == 1)
                p = __uint_as_float(v[c]);
            else
                p = __uint_as_float(v[c]) + __uint_as_float(v[c + 1]) + __uint_as_float(v[c + 2]);
            acc[b] = fmaf(sc[b], p, acc[b]);
        }
    }
}

// Tile row held by tensor-memory lane m (the A row an MMA reads): row
// 8 * i + j, with the 8 lanes of every quarter warp taking 8 consecutive i of
// one j. Row 8i + j sits in box j at slot i, so those 8 lanes read 8 different
// slots, RS = 16 * odd bytes apart: a 16-byte shared load of theirs touches 8
// different bank groups.
__device__ __forceinline__ int tc_lane_row(int m) {
    const int l = m & 31, wq = m >> 5;
    const int i = (l & 7) + 8 * (wq & 1);
    const int j = (l >> 3) + 4 * (wq >> 1);
    return 8 * i + j;
}

// Shared address of tile row r's slot in a raw stage (16-byte aligned), and
// the row segment's offset from it (`lead`, the distance from the 16-byte
// boundary below the segment).
template <int FMT, int NB, int S>
__device__ __forceinline__ uint32_t tc_row_slot(const TcmvArgs& a, uint32_t stage, int64_t tile, int r,
                                                int64_t koff, uint32_t& lead) {
    using L = TcLayout<FMT, NB, S>;
    const int64_t n = tile * 128 + r;
    lead = static_cast<uint32_t>((n * a.rowbytes + koff) & 15);
    if (n < a.n8) return stage + (r & 7) * L::BOXP + (r >> 3) * TcF<FMT>::RS;
    return stage + L::TAIL + static_cast<uint32_t>(min(n - a.n8, static_cast<int64_t>(7))) * TcF<FMT>::RS;
}

// ------------------------------------------------------------ work walk
// Items are (tile, piece); a piece is a run of stages. Every role walks the
// same sequence of (item, stage) pairs, so stage k of the walk uses raw slot
// k % NR in every role.
struct TcItem {
    int m;  // the group's matrix
    int64_t tile, piece, s0, s1;
};

__device__ __forceinline__ TcItem tc_item(const TcmvGroup& g, int64_t item) {
    TcItem it;
    it.m = 0;
    for (int m = 1; m < g.nmat; ++m)
        if (item >= g.m[m].item0) it.m = m;
    const TcmvArgs& a = g.m[it.m];
    const int64_t local = item - a.item0;
    it.tile = local % a.tiles;
    it.piece = local / a.tiles;
    it.s0 = it.piece * a.sps;
    it.s1 = min(it.s0 + a.sps, a.nst);
    return it;
}

// Gathers stage s of the bf16 activations into its B operand slot with
// 16-byte asynchronous copies; every lane then arrives on `bar` (without
// counting itself in) once its copies have landed, so the producer never
// waits for them. Piece u = lane + 32 j is (column c, k octet o, K16 step t)
// with c = u % NB, o = (u / NB) % 2, t = u / (2 NB): the 8 activations of
// batch row c at the stage's position of step t, into row (i % G) * NC + c of
// the step's operand (i = the step's scale group). Columns at or past B are
// never written (zeroed once); pieces past K are zero-filled.
template <int FMT, int NB>
__device__ __forceinline__ void tc_gather_x_stage(const TcmvArgs& a, int64_t s, uint32_t xslot, int lane,
                                                  uint32_t bar) {
    using L = TcLayout<FMT, NB, 1>;
    using F = TcF<FMT>;
    constexpr int NC = L::NC, G = L::G, NCOL = L::NCOL, SPG = F::GK / 16;
    static_assert(32 % NB == 0, "batch bucket");
    const int c = lane % NB;
    if (c < a.B) {
        const uint16_t* xrow = static_cast<const uint16_t*>(a.x) + c * a.K + s * kTcStageK;
        const int64_t krem = a.K - s * kTcStageK;  // K left from the stage start
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int q = lane / NB + j * (32 / NB);
            const int o = q & 1, t = q >> 1;
            const int i = t / SPG, kk = t % SPG;
            const int k = tc_group_k<FMT>(i >> 2, i & 3) + 16 * kk + 8 * o;
            const bool in = k < krem;
            const int row = (i % G) * NC + c;
            const uint32_t dst = xslot + static_cast<uint32_t>(t * NCOL * 32) +
                                 static_cast<uint32_t>(((row >> 3) * 2 + o) * 128 + (row & 7) * 16);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
                         "l"(in ? xrow + k : xrow), "r"(in ? 16 : 0)
                         : "memory");
        }
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------ the kernel

template <int FMT, bool Q8, int NB, int S>
__global__ void __launch_bounds__(kTcThreads, 1)
    tcmv_kernel(const __grid_constant__ TcmvGroup g) {
    using F = TcF<FMT>;
    using L = TcLayout<FMT, NB, S>;
    constexpr int NCOL = L::NCOL;
    constexpr int NR = L::NR, NX = L::NX, NSC = L::NSC, NW = L::NW;
    constexpr uint32_t IDESC = tc::idesc_bf16(128, NCOL);
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const uint32_t b_rfull = sb + L::BARS;
    const uint32_t b_rempty = b_rfull + 8 * NR;
    const uint32_t b_xfull = b_rempty + 8 * NR;
    const uint32_t b_xempty = b_xfull + 8 * NX;
    const uint32_t b_sfull = b_xempty + 8 * NX;
    const uint32_t b_sempty = b_sfull + 8 * NSC;
    const uint32_t b_afull = b_sempty + 8 * NSC;
    const uint32_t b_aempty = b_afull + 8 * 2 * L::NAH;
    const uint32_t b_dfull = b_aempty + 8 * 2 * L::NAH;
    const uint32_t b_dempty = b_dfull + 8 * NW;
    const uint32_t b_final = b_dempty + 8 * NW;
    const uint32_t flag = sb + L::ABORT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = g.st.err;

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (threadIdx.x == 0) {
        for (int r = 0; r < NR; ++r) {
            mbar_init(b_rfull + 8 * r, 1);
            mbar_init(b_rempty + 8 * r, 8);  // the 8 warps of the decode set
        }
        for (int r = 0; r < NX; ++r) {
            // bf16 float mode: one arrival per producer lane, when its copies land
            mbar_init(b_xfull + 8 * r, !Q8 && S == 1 ? 32 : 1);
            mbar_init(b_xempty + 8 * r, 1);  // the MMA commit
        }
        for (int r = 0; r < NSC; ++r) {
            mbar_init(b_sfull + 8 * r, 8);
            mbar_init(b_sempty + 8 * r, 4);
        }
        for (int q = 0; q < 2 * L::NAH; ++q) {  // [set][half slot]
            mbar_init(b_afull + 8 * q, 8);
            mbar_init(b_aempty + 8 * q, 1);
        }
        for (int q = 0; q < NW; ++q) {
            mbar_init(b_dfull + 8 * q, 1);
            mbar_init(b_dempty + 8 * q, 4);
        }
        mbar_init(b_final, 2);  // one commit per MMA issuer
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(flag), "r"(0u) : "memory");
        fence_mbar_init();
    }
    // warps: 0-15 decode (set = warp / 8, part = warp / 4 % 2), 16-19 drain,
    // 20 weight producer, 21-22 MMA issue, 23 activation producer
    constexpr int kDrain0 = 16, kProdW = 20, kMma0 = 21, kProdX = 23;
    if (warp == kMma0) tc::alloc(sb + L::TSLOT, 512);
    if constexpr (!Q8 && S == 1) {
        // bf16 float mode: the rows of the activation slots that no stage
        // writes stay zero
        for (uint32_t u = threadIdx.x; u < NX * L::XT / 16; u += blockDim.x)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sb + L::XOFF + 16 * u), "r"(0u)
                         : "memory");
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = lds_u32(sb + L::TSLOT);

    if (warp == kProdW) {
        // ---------------------------------------------------- raw producer
        // Weights only: they are constant, so no wait for the kernel that
        // precedes this one.
        uint32_t sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
            const TcItem it = tc_item(g, item);
            const TcmvArgs& a = g.m[it.m];
            const int64_t tb16 = a.total_bytes & ~static_cast<int64_t>(15);
            for (int64_t s = it.s0; s < it.s1; ++s, ++sc) {
                const uint32_t slot = sc % NR;
                if (sc >= static_cast<uint32_t>(NR) &&
                    !tcmv_wait_warp(b_rempty + 8 * slot, ((sc / NR) - 1) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t dst0 = sb + slot * L::RAW;
                const uint32_t bar = b_rfull + 8 * slot;
                const int64_t kb0 = s * F::BPS;
                const int64_t koff = kb0 * F::BB;  // byte offset of the stage within a row
                const int64_t len = min(static_cast<int64_t>(F::BPS), a.nb - kb0) * F::BB;
                const int64_t row0 = it.tile * 128;
                const bool boxes = row0 < a.n8;
                // rows past the last whole group of 8 (last tile only): 1-D copies
                // from the 16-byte boundary at or below each row segment, and plain
                // loads for bytes past the last 16-byte boundary of W
                uint32_t bytes = 0;
                int64_t cs = 0, ce = 0;
                int tr = -1;
                {
                    const int64_t n = a.n8 + lane;
                    if (lane < 8 && n < a.N && n >= row0 && n < row0 + 128) {
                        tr = lane;
                        const int64_t st = n * a.rowbytes + koff;
                        const int64_t s16 = st & ~static_cast<int64_t>(15);
                        const int64_t e16 = min((st + len + 15) & ~static_cast<int64_t>(15), tb16);
                        if (e16 > s16) {
                            cs = s16;
                            ce = e16;
                            bytes = static_cast<uint32_t>(e16 - s16);
                        }
                        for (int64_t q = max(e16, s16); q < st + len; ++q)
                            sts_u8(dst0 + L::TAIL + tr * F::RS + static_cast<uint32_t>(q - s16), a.W[q]);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(bar, bytes + (boxes ? 8u * 16u * F::RS : 0u));
                __syncwarp();
                if (boxes && lane < 8) {
                    // box j: row j of the 16 groups of 8 rows of this tile
                    const int64_t xb = (lane * a.rowbytes + koff) & ~static_cast<int64_t>(15);
                    tma_load_2d(dst0 + lane * L::BOXP, &g.map[it.m], static_cast<int>(xb / 2),
                                static_cast<int>(it.tile * 16), bar);
                }
                if (ce > cs)
                    bulk_g2s(dst0 + L::TAIL + tr * F::RS, a.W + cs, static_cast<uint32_t>(ce - cs), bar);
                if (lane == 0) TCMV_TRACE(0, sc);
            }
        }
        // wait (bounded) for the copies still in flight before leaving
        for (uint32_t u = sc > static_cast<uint32_t>(NR) ? sc - NR : 0; u < sc; ++u)
            (void)tcmv_wait_warp(b_rfull + 8 * (u % NR), (u / NR) & 1u, flag, err);
    } else if (warp == kProdX) {
        // ---------------------------------------------------- activation producer
        // bf16 float mode gathers each stage's B operand from the activations
        // (the rows that hold activations are rewritten per stage, all other
        // rows were zeroed at the start); fp32 float mode and q8 mode copy the operand
        // that the preceding kernel prepared (with the exact three-way split
        // or the quantization).
        constexpr bool GATHER = !Q8 && S == 1;
        grid_dependency_wait();  // the activations come from the previous kernel
        uint32_t sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
            const TcItem it = tc_item(g, item);
            const TcmvArgs& a = g.m[it.m];
            for (int64_t s = it.s0; s < it.s1; ++s, ++sc) {
                const uint32_t slot = sc % NX;
                if (sc >= static_cast<uint32_t>(NX) &&
                    !tcmv_wait_warp(b_xempty + 8 * slot, ((sc / NX) - 1) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t bar = b_xfull + 8 * slot, dst = sb + L::XOFF + slot * L::XT;
                if constexpr (GATHER) {
                    tc_gather_x_stage<FMT, NB>(a, s, dst, lane, bar);
                } else if (lane == 0) {
                    mbar_arrive_expect_tx(bar, L::XT);
                    bulk_g2s(dst, a.xt + s * (NCOL * kTcStageK), L::XT, bar);
                }
                __syncwarp();
            }
        }
        for (uint32_t u = sc > static_cast<uint32_t>(NX) ? sc - NX : 0; u < sc; ++u)
            (void)tcmv_wait_warp(b_xfull + 8 * (u % NX), (u / NX) & 1u, flag, err);
    } else if (warp == kMma0 || warp == kMma0 + 1) {
        // ---------------------------------------------------- MMA issue (set = warp - kMma0)
        const uint32_t myset = static_cast<uint32_t>(warp - kMma0);
        if (lane == 0) {
            uint32_t sc = 0;  // stages walked
            bool ok = true;
            for (int64_t item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
                const TcItem it = tc_item(g, item);
                const TcmvArgs& a = g.m[it.m];
                for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                    const uint32_t set = sc & 1u;
                    if (set != myset) continue;
                    const uint32_t xslot = sc % NX;
                    const uint32_t wc = (sc >> 1) * L::W;  // this set's earlier windows
                    if (!tcmv_wait_one(b_xfull + 8 * xslot, (sc / NX) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    // bf16 float mode wrote the operand with generic-proxy copies
                    // (and the zero rows with plain stores): order them before the
                    // tensor core's async-proxy reads
                    if constexpr (!Q8 && S == 1) fence_proxy_async_smem();
                    TCMV_TRACE(1, sc);
                    // descriptors and addresses: per-stage bases plus compile-time
                    // offsets, so the issue loop is a run of MMAs. B operand of
                    // K16 step t: NCOL rows x 16 K at t * NCOL * 32 bytes, core
                    // matrices 128 bytes apart along K, 256 between 8-row groups.
                    const uint64_t bdesc0 = tc::smem_desc(sb + L::XOFF + xslot * L::XT, 128, 256);
                    // half stage h of this set's stage ls is the set's half hs =
                    // 2 ls + h, in A slot hs % NAH (use hs / NAH)
                    const uint32_t hs0 = 2 * (sc >> 1);
                    uint32_t abase = 0, aslot = 0;
                    uint32_t dbase = 0, ws = 0;
#pragma unroll
                    for (int i = 0; i < L::GPS; ++i) {
                        if (i == 0 || i == L::GPS / 2) {
                            const uint32_t hs = hs0 + (i == 0 ? 0u : 1u);
                            if (i != 0) tc::commit(b_aempty + 8 * aslot);
                            aslot = set * L::NAH + hs % L::NAH;
                            if (!tcmv_wait_one(b_afull + 8 * aslot, (hs / L::NAH) & 1u, flag, err)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after();
                            // the half's columns start at the slot; group i's offset
                            // within its stage is taken relative to the half
                            abase = tmem + aslot * (L::SA / 2) - (i == 0 ? 0u : L::SA / 2);
                        }
                        if (i % L::G == 0) {
                            const uint32_t wg = wc + i / L::G;
                            ws = set * L::NWS + wg % L::NWS;
                            if (wg >= static_cast<uint32_t>(L::NWS) &&
                                !tcmv_wait_one(b_dempty + 8 * ws, ((wg / L::NWS) - 1) & 1u, flag, err)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after();
                            dbase = tmem + L::DCOL0 + ws * NCOL;
                        }
                        const uint32_t acol = abase + (i >> 2) * L::QA + F::GA * (i & 3);
#pragma unroll
                        for (int kk = 0; kk < F::GK / 16; ++kk) {
                            const int t = i * (F::GK / 16) + kk;
                            tc::mma_ts(dbase, acol + 8 * kk,
                                       bdesc0 + static_cast<uint64_t>((t * NCOL * 32) >> 4), IDESC,
                                       (i % L::G != 0 || kk > 0) ? 1u : 0u);
                        }
                        if (i % L::G == L::G - 1 || i == L::GPS - 1) tc::commit(b_dfull + 8 * ws);
                    }
                    tc::commit(b_aempty + 8 * aslot);
                    tc::commit(b_xempty + 8 * xslot);
                    TCMV_TRACE(2, sc);
                }
            }
            // every MMA of this CTA has completed before the memory is freed
            tc::commit(b_final);
            (void)tcmv_wait_one(b_final, 0, flag, err);
        }
        __syncwarp();
    } else if (warp < kDrain0) {
        // ---------------------------------------------------- decode (set = warp / 4)
        const uint32_t myset = static_cast<uint32_t>(warp >> 3);
        const int part = (warp >> 2) & 1;
        const int m = 32 * (warp & 3) + lane;
        const int r = tc_lane_row(m);
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        uint32_t sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
            const TcItem it = tc_item(g, item);
            const TcmvArgs& a = g.m[it.m];
            for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                if ((sc & 1u) != myset) continue;
                const uint32_t slot = sc % NR, sslot = sc % NSC;
                if (!tcmv_wait_warp(b_rfull + 8 * slot, (sc / NR) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const int64_t kb0 = s * F::BPS;
                const int nblk = static_cast<int>(min(static_cast<int64_t>(F::BPS), a.nb - kb0));
                uint32_t lead;
                const uint32_t rslot =
                    tc_row_slot<FMT, NB, S>(a, sb + slot * L::RAW, it.tile, r, kb0 * F::BB, lead);
                if ((warp & 7) == 0 && lane == 0) TCMV_TRACE(3, sc);
                // the group scales, for the drainers
                if (sc >= static_cast<uint32_t>(NSC) &&
                    !tcmv_wait_warp(b_sempty + 8 * sslot, ((sc / NSC) - 1) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                tc_store_scales<FMT>(rslot + lead, nblk, sb + L::SOFF + sslot * L::SCB, m, part);
                __syncwarp();
                if (lane == 0) mbar_arrive(b_sfull + 8 * sslot);
                // each half of the set's A stage, once its previous contents
                // have been read by their MMAs: the MMAs of one half run while
                // the other half is decoded
                const uint32_t ls = sc >> 1;
                const bool uni = a.rowbytes % 16 == 0;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    // the set's half hs = 2 ls + h goes to A slot hs % NAH, once the
                    // MMAs of the slot's previous half have read it
                    const uint32_t hs = 2 * ls + h;
                    const uint32_t ab = myset * L::NAH + hs % L::NAH;
                    if (hs >= static_cast<uint32_t>(L::NAH) &&
                        !tcmv_wait_warp(b_aempty + 8 * ab, ((hs / L::NAH) - 1) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t acol = lane_base + ab * (L::SA / 2) - static_cast<uint32_t>(h) * (L::SA / 2);
                    tc_decode_half<FMT>(rslot, lead, uni, acol, h, part);
                    tc::wait_st();
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_afull + 8 * ab);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_rempty + 8 * slot);
                if ((warp & 7) == 0 && lane == 0) TCMV_TRACE(4, sc);
            }
        }
    } else {
        // ---------------------------------------------------- drain (warps 8-11)
        const int m = 32 * (warp & 3) + lane;
        const int r = tc_lane_row(m);
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        grid_dependency_wait();  // y, the partial sums and the activation scales
        uint32_t sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
            const TcItem it = tc_item(g, item);
            const TcmvArgs& a = g.m[it.m];
            const int64_t n = it.tile * 128 + r;
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
            for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                const uint32_t sslot = sc % NSC;
                if (!tcmv_wait_warp(b_sfull + 8 * sslot, (sc / NSC) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t scales = sb + L::SOFF + sslot * L::SCB;
                const uint32_t set = sc & 1u;
#pragma unroll 1
                for (int w = 0; w < L::W; ++w) {
                    const uint32_t wc = (sc >> 1) * L::W + w;  // the set's window count
                    const uint32_t ws = set * L::NWS + wc % L::NWS;
                    if (!tcmv_wait_warp(b_dfull + 8 * ws, (wc / L::NWS) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    if (warp == kDrain0 && lane == 0) TCMV_TRACE(5, wc);
                    tc::fence_after();
                    tc_drain_window<FMT, NB, S, Q8>(lane_base + L::DCOL0 + ws * NCOL, scales, m, w,
                                                    s * (kTcStageK / 32), a, acc);
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_dempty + 8 * ws);
                    if (warp == kDrain0 && lane == 0) TCMV_TRACE(6, wc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_sempty + 8 * sslot);
            }
            if (ok && n < a.N) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b >= a.B) break;
                    if (a.pieces == 1)
                        a.y[b * a.N + n] = acc[b];
                    else
                        a.part[(it.piece * a.B + b) * a.N + n] = acc[b];
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == kMma0) {
        tc::fence_after();
        tc::dealloc(tmem, 512);
    }
}

template <int FMT>
TcmvKernel tcmv_pick(bool q8, int NB, int S) {
    if (q8) {
        if (S != 1) return nullptr;
        switch (NB) {
            case 1: return tcmv_kernel<FMT, true, 1, 1>;
            case 2: return tcmv_kernel<FMT, true, 2, 1>;
            case 4: return tcmv_kernel<FMT, true, 4, 1>;
            case 8: return tcmv_kernel<FMT, true, 8, 1>;
            case 16: return tcmv_kernel<FMT, true, 16, 1>;
        }
        return nullptr;
    }
    if (S == 1) {
        switch (NB) {
            case 1: return tcmv_kernel<FMT, false, 1, 1>;
            case 2: return tcmv_kernel<FMT, false, 2, 1>;
            case 4: return tcmv_kernel<FMT, false, 4, 1>;
            case 8: return tcmv_kernel<FMT, false, 8, 1>;
            case 16: return tcmv_kernel<FMT, false, 16, 1>;
        }
    } else if (S == 3) {
        switch (NB) {
            case 1: return tcmv_kernel<FMT, false, 1, 3>;
            case 2: return tcmv_kernel<FMT, false, 2, 3>;
            case 4: return tcmv_kernel<FMT, false, 4, 3>;
            case 8: return tcmv_kernel<FMT, false, 8, 3>;
            case 16: return tcmv_kernel<FMT, false, 16, 3>;
        }
    }
    return nullptr;
}

template <int FMT>
uint32_t tcmv_smem_of(int NB, int S) {
#define QMM_TC_SMEM(nb, s) \
    if (NB == nb && S == s) return TcLayout<FMT, nb, s>::SMEM;
    QMM_TC_SMEM(1, 1) QMM_TC_SMEM(2, 1) QMM_TC_SMEM(4, 1) QMM_TC_SMEM(8, 1) QMM_TC_SMEM(16, 1)
    QMM_TC_SMEM(1, 3) QMM_TC_SMEM(2, 3) QMM_TC_SMEM(4, 3) QMM_TC_SMEM(8, 3) QMM_TC_SMEM(16, 3)
#undef QMM_TC_SMEM
    return 0;
}

}  // namespace qmm
