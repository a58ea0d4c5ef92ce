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
// CTA (448 threads, one per SM, persistent over work items = 128-row tile x
// a range of 256-wide K stages):
//   warps 0-7   decode weights -> A; two sets of 4 warps take alternate
//               stages (row = 32 * (warp % 4) + lane)
//   warps 8-11  drain D: load the accumulators, apply the scales read from
//               the raw stage, sum, store
//   warp 12     producer: per stage, 8 tensor-map copies of the tile's raw
//               blocks (W seen as rows of 8 weight rows: any row pitch becomes a
//               16-byte multiple, and one copy brings row j of 16 such groups),
//               1-D bulk copies for the rows past the last whole group of 8,
//               and one 1-D bulk copy of the stage's activation tile
//   warp 13     owns the tensor memory; lane 0 issues the MMAs
// Rings: raw stages (producer -> decoders, drainers, MMA), A slots per
// decode set (decoders -> MMA), D slots (MMA -> drainers), each with a
// full / empty mbarrier pair, every wait bounded in time.
#pragma once

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
    static constexpr int NCOL = NC <= 16 ? 16 : (NC <= 32 ? 32 : 48);  // MMA N
};

template <int FMT, int NB, int S>
struct TcLayout {
    using F = TcF<FMT>;
    static constexpr int NCOL = TcCols<NB, S>::NCOL;
    // raw part of a stage: 8 boxes (row j of every group of 8 rows, 16 groups
    // per tile), rows one slot RS apart, then a tail area for the up to 7
    // rows past the last whole group of 8; tensor-map destinations are
    // 128-byte aligned
    static constexpr uint32_t BOXP = 16u * F::RS;
    static_assert(BOXP % 128 == 0 && (8u * F::RS) % 128 == 0, "box alignment");
    static constexpr uint32_t TAIL = 8 * BOXP;
    static constexpr uint32_t RAW = TAIL + 8u * F::RS;
    static constexpr uint32_t XT = static_cast<uint32_t>(NCOL) * kTcStageK * 2;
    static constexpr uint32_t STAGE = RAW + XT;
    static constexpr int QA = 4 * F::GA;                       // A columns per quad
    static constexpr int NAH = (FMT != FMT_Q6_K && NCOL == 48) ? 1 : 2;  // A slots per set
    static constexpr int NA = 2 * NAH;
    static constexpr int ND = NCOL == 16 ? 4 : 2;              // D slots (quads)
    static constexpr uint32_t DCOL0 = NA * QA;                 // first D column
    static constexpr uint32_t TNEED = DCOL0 + ND * 4 * NCOL;
    static_assert(TNEED <= 512, "tensor memory");
    // barriers: raw_full[NR], raw_empty[NR], a_full[NA], a_empty[NA],
    // d_full[ND], d_empty[ND], final
    static constexpr int NR0 = static_cast<int>((kTcSmemCap - 512) / STAGE);
    static constexpr int NR = NR0 > 6 ? 6 : NR0;               // raw stages in flight
    static_assert(NR >= 3, "raw stages");
    static constexpr uint32_t BARS = NR * STAGE;
    static constexpr uint32_t NBARS = 2 * NR + 2 * NA + 2 * ND + 1;
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
// Warp-collective wait that also gives up once another role of the CTA gave
// up; every lane leaves with the same answer (the tensor-memory operations
// that follow are .sync.aligned).
__device__ __forceinline__ bool tcmv_wait_warp(uint32_t bar, uint32_t parity, uint32_t flag,
                                               unsigned int* err) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((it & 63u) == 0) {
            int give_up = lds_u32(flag) != 0 ? 1 : 0;
            if (!give_up && globaltimer_ns() - t0 > kWaitLimitNs) give_up = 2;
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
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
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

// ------------------------------------------------------------ decode a quad
// Writes the A operand of the 4 groups of quad Q of this thread's row into
// tensor-memory columns `acol` (lane = this row).
template <int FMT>
__device__ __forceinline__ void tc_decode_quad(uint32_t rowp, int Q, uint32_t acol) {
    using F = TcF<FMT>;
    if constexpr (FMT == FMT_Q6_K) {
        uint32_t qh[4], qa[4], qb[4];
        lds_words_unaligned<4>(rowp + 128 + 16 * Q, qh);
        lds_words_unaligned<4>(rowp + 16 * Q, qa);
        lds_words_unaligned<4>(rowp + 64 + 16 * Q, qb);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            // group j = Q + 4g: ql run (j & 7), nibble j >> 3, qh field j >> 2 = g
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
            tc::st8(acol + F::GA * g, A);
        }
    } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t blk = rowp + F::BB * (4 * Q + g);
            uint32_t A[16];
            if constexpr (FMT == FMT_Q4_0) {
                uint32_t qs[4];
                lds_words_unaligned<4>(blk + 2, qs);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t lo = qs[w] & 0x0F0F0F0Fu;         // elements 4w..4w+3
                    const uint32_t hi = (qs[w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w..
                    A[2 * w] = bf_add(bf_pair_lo(lo), kBfNeg136);
                    A[2 * w + 1] = bf_add(bf_pair_hi(lo), kBfNeg136);
                    A[8 + 2 * w] = bf_add(bf_pair_lo(hi), kBfNeg136);
                    A[8 + 2 * w + 1] = bf_add(bf_pair_hi(hi), kBfNeg136);
                }
            } else {
                uint32_t qs[8];
                lds_words_unaligned<8>(blk + 2, qs);
#pragma unroll
                for (int w = 0; w < 8; ++w) q8_bf_pairs(qs[w], A[2 * w], A[2 * w + 1]);
            }
            tc::st16(acol + F::GA * g, A);
        }
    }
}

// The 4 group scales of quad Q of this thread's row, read from the raw stage.
// Blocks past the end of the row (last stage of a ragged K) hold stale bytes;
// their activations are zero and their scale is 0.
template <int FMT>
__device__ __forceinline__ void tc_quad_scales(uint32_t rowp, int Q, int nblk, float (&s)[4]) {
    if constexpr (FMT == FMT_Q6_K) {
        const float d = half_bits_to_float(lds_u16(rowp + 208));
#pragma unroll
        for (int g = 0; g < 4; ++g) s[g] = d * static_cast<float>(lds_s8(rowp + 192 + Q + 4 * g));
        (void)nblk;
    } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int i = 4 * Q + g;
            const float d = half_bits_to_float(lds_u16(rowp + TcF<FMT>::BB * i));
            s[g] = i < nblk ? d : 0.0f;
        }
    }
}

// ------------------------------------------------------------ drain a quad
// Loads the 4 accumulators of a quad (this thread's row) and adds
// s * (activation scale) * P to acc[b] for every activation row b.
template <int NC>
struct TcLd {
    static constexpr int N = NC <= 1 ? 1 : NC <= 2 ? 2 : NC <= 4 ? 4 : NC <= 8 ? 8 : NC <= 16 ? 16
                             : NC <= 32 ? 32 : 48;
};

template <int NL>
__device__ __forceinline__ void tc_ld_cols(uint32_t taddr, uint32_t (&v)[NL]) {
    if constexpr (NL == 48) {
        tc::ld<32>(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tc::ld<16>(taddr + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
    } else {
        tc::ld<NL>(taddr, v);
    }
}

template <int NB, int S, bool Q8>
__device__ __forceinline__ void tc_drain_use(const uint32_t* v, float s, int64_t xblk,
                                             const TcmvArgs& a, float (&acc)[NB]) {
    float sc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) sc[b] = s;
    if constexpr (Q8) {
        // activation scales of this 32-block, stored [block][NB]
        const float* xs = a.xs + xblk * NB;
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
        float p;
        if constexpr (S == 1)
            p = __uint_as_float(v[b]);
        else
            p = __uint_as_float(v[3 * b]) + __uint_as_float(v[3 * b + 1]) +
                __uint_as_float(v[3 * b + 2]);
        acc[b] = fmaf(sc[b], p, acc[b]);
    }
}

template <int NB, int S, bool Q8, int FMT>
__device__ __forceinline__ void tc_drain_quad(uint32_t dcol, uint32_t rowp, int Q, int nblk,
                                              int64_t xblk0, const TcmvArgs& a, float (&acc)[NB]) {
    constexpr int NCOL = TcCols<NB, S>::NCOL;
    constexpr int NL = TcLd<NB * S>::N;
    float s[4];
    if constexpr (NB * S <= 16) {
        // all four loads in flight, the scales read meanwhile, one wait
        uint32_t v[4][NL];
#pragma unroll
        for (int g = 0; g < 4; ++g) tc_ld_cols<NL>(dcol + NCOL * g, v[g]);
        tc_quad_scales<FMT>(rowp, Q, nblk, s);
        tc::wait_ld();
#pragma unroll
        for (int g = 0; g < 4; ++g)
            tc_drain_use<NB, S, Q8>(v[g], s[g], xblk0 + tc_group_xblk<FMT>(Q, g), a, acc);
    } else {
        tc_quad_scales<FMT>(rowp, Q, nblk, s);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t v[NL];
            tc_ld_cols<NL>(dcol + NCOL * g, v);
            tc::wait_ld();
            tc_drain_use<NB, S, Q8>(v, s[g], xblk0 + tc_group_xblk<FMT>(Q, g), a, acc);
        }
    }
}

// ------------------------------------------------------------ tensor-map copy
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared address of row m's data in a raw stage (lead = the row segment's
// offset from the 16-byte boundary below it).
template <int FMT, int NB, int S>
__device__ __forceinline__ uint32_t tc_row_ptr(const TcmvArgs& a, uint32_t stage, int64_t tile, int m,
                                               int64_t koff) {
    using L = TcLayout<FMT, NB, S>;
    const int64_t n = tile * 128 + m;
    const uint32_t lead = static_cast<uint32_t>((n * a.rowbytes + koff) & 15);
    if (n < a.n8) return stage + (m & 7) * L::BOXP + (m >> 3) * TcF<FMT>::RS + lead;
    return stage + L::TAIL + static_cast<uint32_t>(min(n - a.n8, static_cast<int64_t>(7))) * TcF<FMT>::RS +
           lead;
}

// ------------------------------------------------------------ work walk
// Items are (tile, piece); a piece is a run of stages. Every role walks the
// same sequence of (item, stage) pairs, so stage k of the walk uses raw slot
// k % NR in every role.
struct TcItem {
    int64_t tile, piece, s0, s1;
};

__device__ __forceinline__ TcItem tc_item(const TcmvArgs& a, int64_t item) {
    TcItem it;
    it.tile = item % a.tiles;
    it.piece = item / a.tiles;
    it.s0 = it.piece * a.sps;
    it.s1 = min(it.s0 + a.sps, a.nst);
    return it;
}

// ------------------------------------------------------------ the kernel

template <int FMT, bool Q8, int NB, int S>
__global__ void __launch_bounds__(kTcThreads, 1)
    tcmv_kernel(const TcmvArgs a, const __grid_constant__ CUtensorMap tmap) {
    using F = TcF<FMT>;
    using L = TcLayout<FMT, NB, S>;
    constexpr int NCOL = L::NCOL;
    constexpr int NR = L::NR, NA = L::NA, NAH = L::NAH, ND = L::ND;
    constexpr uint32_t IDESC = tc::idesc_bf16(128, NCOL);
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const uint32_t b_rfull = sb + L::BARS;
    const uint32_t b_rempty = b_rfull + 8 * NR;
    const uint32_t b_afull = b_rempty + 8 * NR;
    const uint32_t b_aempty = b_afull + 8 * NA;
    const uint32_t b_dfull = b_aempty + 8 * NA;
    const uint32_t b_dempty = b_dfull + 8 * ND;
    const uint32_t b_final = b_dempty + 8 * ND;
    const uint32_t flag = sb + L::ABORT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = a.st.err;

    grid_launch_dependents();
    live_bump(a.st, a.live_slot);
    if (threadIdx.x == 0) {
        for (int r = 0; r < NR; ++r) {
            mbar_init(b_rfull + 8 * r, 1);
            mbar_init(b_rempty + 8 * r, 9);  // 4 decoders + 4 drainers + the MMA commit
        }
        for (int q = 0; q < NA; ++q) {
            mbar_init(b_afull + 8 * q, 4);
            mbar_init(b_aempty + 8 * q, 1);
        }
        for (int q = 0; q < ND; ++q) {
            mbar_init(b_dfull + 8 * q, 1);
            mbar_init(b_dempty + 8 * q, 4);
        }
        mbar_init(b_final, 1);
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(flag), "r"(0u) : "memory");
        fence_mbar_init();
    }
    if (warp == 13) tc::alloc(sb + L::TSLOT, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = lds_u32(sb + L::TSLOT);

    if (warp == 12) {
        // ---------------------------------------------------- producer
        const int64_t tb16 = a.total_bytes & ~static_cast<int64_t>(15);
        uint32_t issued = 0;
        bool waited = false, ok = true;
        int64_t pend[NR];
        int npend = 0;
        auto issue_x = [&](uint32_t slot, int64_t s) {
            if (lane == 0)
                bulk_g2s(sb + slot * L::STAGE + L::RAW, a.xt + s * (NCOL * kTcStageK), L::XT,
                         b_rfull + 8 * slot);
        };
        for (int64_t item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
            const TcItem it = tc_item(a, item);
            for (int64_t s = it.s0; s < it.s1; ++s) {
                const uint32_t slot = issued % NR;
                if (issued >= static_cast<uint32_t>(NR) &&
                    !tcmv_wait_warp(b_rempty + 8 * slot, ((issued / NR) - 1) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t dst0 = sb + slot * L::STAGE;
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
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, bytes + L::XT + (boxes ? 8u * 16u * F::RS : 0u));
                __syncwarp();
                if (boxes && lane < 8) {
                    // box j: row j of the 16 groups of 8 rows of this tile
                    const int64_t xb = (lane * a.rowbytes + koff) & ~static_cast<int64_t>(15);
                    tma_load_2d(dst0 + lane * L::BOXP, &tmap, static_cast<int>(xb / 2),
                                static_cast<int>(it.tile * 16), bar);
                }
                if (ce > cs)
                    bulk_g2s(dst0 + L::TAIL + tr * F::RS, a.W + cs, static_cast<uint32_t>(ce - cs), bar);
                if (lane == 0) TCMV_TRACE(0, issued);
                if (waited)
                    issue_x(slot, s);
                else
                    pend[npend++] = s;
                ++issued;
                // the weights of the first stages go out before waiting for the
                // kernel that wrote the activation tile
                if (!waited && issued == static_cast<uint32_t>(NR)) {
                    grid_dependency_wait();
                    waited = true;
                    for (int p = 0; p < npend; ++p) issue_x(static_cast<uint32_t>(p), pend[p]);
                    npend = 0;
                }
            }
        }
        if (!waited) {
            grid_dependency_wait();
            for (int p = 0; p < npend; ++p) issue_x(static_cast<uint32_t>(p), pend[p]);
        }
        // wait (bounded) for the copies still in flight before leaving
        for (uint32_t u = issued > static_cast<uint32_t>(NR) ? issued - NR : 0; u < issued; ++u)
            (void)tcmv_wait_warp(b_rfull + 8 * (u % NR), (u / NR) & 1u, flag, err);
    } else if (warp == 13) {
        // ---------------------------------------------------- MMA issue
        if (lane == 0) {
            uint32_t qc = 0, sc = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
                const TcItem it = tc_item(a, item);
                for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                    const uint32_t slot = sc % NR;
                    const uint32_t set = sc & 1u;
                    if (!tcmv_wait_one(b_rfull + 8 * slot, (sc / NR) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    TCMV_TRACE(1, sc);
                    const uint32_t xaddr = sb + slot * L::STAGE + L::RAW;
#pragma unroll 1
                    for (int Q = 0; Q < F::QPS; ++Q, ++qc) {
                        const uint32_t lq = (sc >> 1) * F::QPS + Q;  // quad count of the set
                        const uint32_t as = set * NAH + lq % NAH;
                        const uint32_t ds = qc % ND;
                        if (!tcmv_wait_one(b_afull + 8 * as, (lq / NAH) & 1u, flag, err) ||
                            (qc >= static_cast<uint32_t>(ND) &&
                             !tcmv_wait_one(b_dempty + 8 * ds, ((qc / ND) - 1) & 1u, flag, err))) {
                            ok = false;
                            break;
                        }
                        TCMV_TRACE(7, qc);
                        tc::fence_after();
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const uint32_t dcol = tmem + L::DCOL0 + ds * 4 * NCOL + NCOL * g;
                            const uint32_t acol = tmem + as * L::QA + F::GA * g;
                            const int k0 = tc_group_k<FMT>(Q, g);
#pragma unroll
                            for (int kk = 0; kk < F::GK / 16; ++kk) {
                                const uint64_t bd = tc::smem_desc(
                                    xaddr + static_cast<uint32_t>((k0 / 8 + 2 * kk) * 128), 128,
                                    kTcStageK / 8 * 128);
                                tc::mma_ts(dcol, acol + 8 * kk, bd, IDESC, kk > 0 ? 1u : 0u);
                            }
                        }
                        tc::commit(b_aempty + 8 * as);
                        tc::commit(b_dfull + 8 * ds);
                    }
                    tc::commit(b_rempty + 8 * slot);
                    TCMV_TRACE(2, sc);
                }
            }
            // every MMA of this CTA has completed before the memory is freed
            tc::commit(b_final);
            (void)tcmv_wait_one(b_final, 0, flag, err);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ---------------------------------------------------- decode (set = warp / 4)
        const uint32_t myset = static_cast<uint32_t>(warp >> 2);
        const int m = 32 * (warp & 3) + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        uint32_t sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
            const TcItem it = tc_item(a, item);
            for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                if ((sc & 1u) != myset) continue;
                const uint32_t slot = sc % NR;
                if (!tcmv_wait_warp(b_rfull + 8 * slot, (sc / NR) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t rowp = tc_row_ptr<FMT, NB, S>(a, sb + slot * L::STAGE, it.tile, m,
                                                             s * F::BPS * F::BB);
                if ((warp & 3) == 0 && lane == 0) TCMV_TRACE(3, sc);
#pragma unroll 1
                for (int Q = 0; Q < F::QPS; ++Q) {
                    const uint32_t lq = (sc >> 1) * F::QPS + Q;
                    const uint32_t as = myset * NAH + lq % NAH;
                    if (lq >= static_cast<uint32_t>(NAH) &&
                        !tcmv_wait_warp(b_aempty + 8 * as, ((lq / NAH) - 1) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    tc_decode_quad<FMT>(rowp, Q, lane_base + as * L::QA);
                    tc::wait_st();
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_afull + 8 * as);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_rempty + 8 * slot);
                if ((warp & 3) == 0 && lane == 0) TCMV_TRACE(4, sc);
            }
        }
    } else {
        // ---------------------------------------------------- drain
        const int m = 32 * (warp & 3) + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        grid_dependency_wait();  // y, the partial sums and the activation scales
        uint32_t qc = 0, sc = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
            const TcItem it = tc_item(a, item);
            const int64_t n = it.tile * 128 + m;
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
            for (int64_t s = it.s0; ok && s < it.s1; ++s, ++sc) {
                const uint32_t slot = sc % NR;
                if (!tcmv_wait_warp(b_rfull + 8 * slot, (sc / NR) & 1u, flag, err)) {
                    ok = false;
                    break;
                }
                const int64_t kb0 = s * F::BPS;
                const int nblk = static_cast<int>(min(static_cast<int64_t>(F::BPS), a.nb - kb0));
                const uint32_t rowp = tc_row_ptr<FMT, NB, S>(a, sb + slot * L::STAGE, it.tile, m,
                                                             kb0 * F::BB);
#pragma unroll 1
                for (int Q = 0; Q < F::QPS; ++Q, ++qc) {
                    const uint32_t ds = qc % ND;
                    if (!tcmv_wait_warp(b_dfull + 8 * ds, (qc / ND) & 1u, flag, err)) {
                        ok = false;
                        break;
                    }
                    if (warp == 8 && lane == 0) TCMV_TRACE(5, qc);
                    tc::fence_after();
                    tc_drain_quad<NB, S, Q8, FMT>(lane_base + L::DCOL0 + ds * 4 * NCOL, rowp, Q, nblk,
                                                  s * (kTcStageK / 32), a, acc);
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_dempty + 8 * ds);
                    if (warp == 8 && lane == 0) TCMV_TRACE(6, qc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_rempty + 8 * slot);
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
    if (warp == 13) {
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
