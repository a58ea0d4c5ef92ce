// mvh.cuh -- fused dequantize + matvec for 1..8 bf16 activation rows (float
// mode) on the warp-level tensor-core MMA with fp16 operands, for any mix of
// the three weight formats in one launch:
//
//   y[b][n] = sum_k w[n][k] * x[b][k],   b < B <= 8
//
// The unpack is the cost that matters (quantprobe "LAWS.md", Law 4
// amendment L-15), so each step is chosen for few instructions per weight:
//
// * Weights are the A operand of mma.sync m16n8k16 (fp16, fp32 accumulate):
//   16 weight rows x 16 K. For q6_K the sub-block scale is folded into A:
//   sc * (q - 32) is an integer of magnitude <= 62 * 32 < 2048, exact in
//   fp16, made from the fp16 value 1024 + code (one byte-permute per two
//   weights) by ONE fp16x2 FMA, (1024 + c) * sc - 1056 * sc (the bias is an
//   exact fp16 value, and the fused result is exact). The MMA then sums a
//   whole 256-weight super-block into one fp32 accumulator, and d is applied
//   once per super-block. Q4_0 / Q8_0: A = q - 8 / q exactly, d applied once
//   per 32-weight block. A q6_K tile whose scales leave -62..62 takes the
//   exact two-MMA form sc = lo + 8 hi (0 <= lo < 8) instead.
// * Activations are the B operand: the prep kernel (mvh.cu) writes each
//   activation row as fp16 x * 2^e, e chosen per row so that the row's
//   largest magnitude lies in [2^14, 2^15); every bf16 value within a factor
//   2^28 of that maximum is exact in fp16, smaller ones are off by less than
//   2^-38 of it. Outputs are scaled back by 2^-e (exact).
// * K positions inside an MMA are permuted freely (A and B the same way):
//   lane (g = lane / 4, c = lane % 4) feeds 4 consecutive weights per row and
//   MMA. Over the 16 MMAs of a q6_K stage its weights of a row are the scale
//   groups c, c + 4, c + 8, c + 12 (16 consecutive weights each), so its code
//   bytes are three 16-byte runs of ql / qh; Q4_0 / Q8_0: weights 8c .. 8c + 7
//   of each block. Its activations are runs of 16 bytes.
//
// Work item: 32 rows of one matrix at stride 8 (rows j + 8 (G + i), i < 32),
// all of K in stages (q6_K one super-block, Q4_0 8 blocks, Q8_0 4 blocks).
// Rows 8 apart start at the same offset modulo 16 (the pitch of 8 rows is a
// multiple of 16 for every even row size), so the byte lead of a stage is
// the same for all 32 rows of an item and the realignment of the code bytes
// is warp-uniform. A stage arrives by 2-D TMA with W seen as
// [N / 8][8 * rowbytes] 16-bit elements, in boxes 32 rows high that land
// row after row: q6_K four boxes 64 bytes wide (the 14 pieces of 16 bytes a
// super-block and its lead cover, and 2 more), so the 128-bit loads of one
// load phase (rows 2k and 2k + 1, lanes c = 0..3 reading pieces c + s) hit 32
// different banks; Q4_0 / Q8_0 three boxes 48 bytes wide (their 144 bytes
// exactly), read with 32-bit loads. Box destinations are 128-byte aligned.
//
// Each warp streams its own items through a private ring of NS stages (an
// mbarrier per slot, waits bounded in time); a team of KS warps of a CTA may
// share an item (member m takes stages m, m + KS, ...) and add their sums in
// member order at the end (named barrier), so results do not depend on
// timing.
#pragma once

#include <cuda_fp16.h>

#include "kernels.h"

namespace qmm {

constexpr int kMvhNS = 3;
constexpr int kMvhRows = 32;                // rows per item: two 16-row MMA tiles
// box width in bytes and boxes per stage: q6_K 4 x 64, Q4_0 / Q8_0 3 x 48
__host__ __device__ constexpr uint32_t mvh_box_w(int fmt) { return fmt == FMT_Q6_K ? 64u : 48u; }
__host__ __device__ constexpr int mvh_boxes(int fmt) { return fmt == FMT_Q6_K ? 4 : 3; }
constexpr uint32_t kMvhSlot = 4 * 64 * kMvhRows;   // the largest stage: 8 KB
constexpr uint32_t kMvhPartOff = kMvhWarps * kMvhNS * kMvhSlot;  // team sums, after the rings
constexpr uint32_t kMvhBarOff = kMvhPartOff + kMvhWarps * 8 * 32 * 4;
constexpr uint32_t kMvhSmem = kMvhBarOff + kMvhWarps * kMvhNS * 8;
static_assert(kMvhSmem <= 227u * 1024, "shared memory");

// D = A B + C, m16n8k16, fp16 A (row) and B (col), fp32 C and D
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// the fp16 pair (v, v) of a small integer v (exact)
__device__ __forceinline__ uint32_t h2_splat(int v) {
    const uint32_t h = __half_as_ushort(__int2half_rn(v));
    return h | (h << 16);
}

__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// code bytes 0, 1 / 2, 3 of w -> fp16 pairs (1024 + byte)
__device__ __forceinline__ uint32_t h_pair01(uint32_t w) { return __byte_perm(w, 0x64646464u, 0x5140); }
__device__ __forceinline__ uint32_t h_pair23(uint32_t w) { return __byte_perm(w, 0x64646464u, 0x7362); }

constexpr uint32_t kH2M1032 = 0xE408E408u;  // fp16 pair (-1032, -1032): (1024 + q) - 1032 = q - 8
constexpr uint32_t kH2M1056 = 0xE420E420u;  // (-1056, -1056): (1024 + q) - 1056 = q - 32
constexpr uint32_t kH2M1152 = 0xE480E480u;  // (-1152, -1152): (1024 + (v ^ 128)) - 1152 = v, signed byte v

__device__ __forceinline__ void mvh_lds_v4(uint32_t a, uint32_t* w) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(a));
}

// q6_K stage slot: shared address of 16-byte piece p of row r (four boxes of
// [32 rows][64 B], 2 KB apart).
__device__ __forceinline__ uint32_t q6k_piece(uint32_t slot, int r, int p) {
    return slot + static_cast<uint32_t>(p >> 2) * 2048u + 64u * static_cast<uint32_t>(r) +
           16u * static_cast<uint32_t>(p & 3);
}

// The 16 bytes at byte lead L (even, < 16; QW = L / 4 and sel shifts by
// L % 4) of piece p of row r and the next piece.
template <int QW>
__device__ __forceinline__ void mvh_seg(uint32_t slot, int r, int p, uint32_t sel, uint32_t (&o)[4]) {
    uint32_t w[8];
    mvh_lds_v4(q6k_piece(slot, r, p), w);
    mvh_lds_v4(q6k_piece(slot, r, p + 1), w + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __byte_perm(w[QW + i], w[QW + i + 1], sel);
}

// Q4_0 / Q8_0 stage slot: shared address of logical byte o of row r (three
// boxes of [32 rows][48 B], 1536 bytes apart).
__device__ __forceinline__ uint32_t mvh_addr(uint32_t slot, int r, uint32_t o) {
    return slot + (o / 48u) * 1536u + 48u * static_cast<uint32_t>(r) + (o % 48u);
}

// Four bytes at logical byte o of row r; ALIGNED says whether o % 4 == 0
// (else o % 4 == 2, and the word is put together from the aligned words
// around it; an aligned word never straddles two boxes).
template <bool ALIGNED>
__device__ __forceinline__ uint32_t mvh_word(uint32_t slot, int r, uint32_t o) {
    if constexpr (ALIGNED) {
        return lds_u32(mvh_addr(slot, r, o));
    } else {
        const uint32_t o0 = o - 2;
        return __byte_perm(lds_u32(mvh_addr(slot, r, o0)), lds_u32(mvh_addr(slot, r, o0 + 4)), 0x5432);
    }
}

__device__ __forceinline__ float mvh_half(uint32_t slot, int r, uint32_t o) {
    return half_bits_to_float(lds_u16(mvh_addr(slot, r, o)));
}

// ------------------------------------------------------------ q6_K stage
// One 16-row tile: rows ra (lane row g) and rb (g + 8) of the stage. Lane c's
// scale groups are c + 4Q (Q = 0..3): ql bytes 16c .. (Q = 0 low nibble, Q = 2
// high) and 64 + 16c .. (Q = 1 low, Q = 3 high), qh bytes 16c .. (2-bit
// field Q), scale byte c of scale word Q. MMA (Q, u) takes the lane's weights
// 16 (c + 4Q) + 4u .. + 3, whose activations are x[8Q + 2u], x[8Q + 2u + 1].

// code word of the lane's weights 4u .. 4u + 3 of group quad Q
template <int Q>
__device__ __forceinline__ uint32_t q6k_code(const uint32_t (&ql0)[4], const uint32_t (&ql1)[4],
                                             const uint32_t (&qh)[4], int u) {
    const uint32_t l = (Q & 1) ? ql1[u] : ql0[u];
    const uint32_t lo = (Q >> 1) ? (l >> 4) : l;
    const uint32_t hi = Q == 0 ? (qh[u] << 4) : Q == 1 ? (qh[u] << 2) : Q == 2 ? qh[u] : (qh[u] >> 2);
    return (lo & 0x0F0F0F0Fu) | (hi & 0x30303030u);
}

// signed scale byte c of w
__device__ __forceinline__ int q6k_sc(uint32_t w, int c) {
    return static_cast<int>(static_cast<int8_t>(static_cast<uint8_t>(w >> (8 * c))));
}

// Adds the tile's products of one super-block into D (not cleared here).
// Returns false (doing nothing) if a scale of the tile lies outside -62..62.
template <int QW>
__device__ __forceinline__ bool q6k_tile_fast(uint32_t slot, int ra, int rb, int c, uint32_t sel, uint32_t selc,
                                              const uint32_t (&x)[32], float (&D)[4]) {
    uint32_t qa0[4], qa1[4], ha[4], sa[4], qb0[4], qb1[4], hb[4], sb[4];
    mvh_seg<QW>(slot, ra, 12, sel, sa);
    mvh_seg<QW>(slot, rb, 12, sel, sb);
    bool big = false;
#pragma unroll
    for (int Q = 0; Q < 4; ++Q) {
        const int s0 = q6k_sc(sa[Q], c), s1 = q6k_sc(sb[Q], c);
        big = big || s0 > 62 || s0 < -62 || s1 > 62 || s1 < -62;
    }
    if (__any_sync(0xffffffffu, big)) return false;
    mvh_seg<QW>(slot, ra, c, sel, qa0);
    mvh_seg<QW>(slot, ra, 4 + c, sel, qa1);
    mvh_seg<QW>(slot, ra, 8 + c, sel, ha);
    mvh_seg<QW>(slot, rb, c, sel, qb0);
    mvh_seg<QW>(slot, rb, 4 + c, sel, qb1);
    mvh_seg<QW>(slot, rb, 8 + c, sel, hb);
#define QMM_MVH_Q6K_QUAD(Q)                                                                     \
    {                                                                                           \
        const uint32_t s2a = h2_add(__byte_perm(sa[Q] ^ 0x80808080u, 0x64646464u, selc), kH2M1152); \
        const uint32_t s2b = h2_add(__byte_perm(sb[Q] ^ 0x80808080u, 0x64646464u, selc), kH2M1152); \
        const uint32_t b2a = h2_mul(s2a, kH2M1056), b2b = h2_mul(s2b, kH2M1056);                \
        _Pragma("unroll") for (int u = 0; u < 4; ++u) {                                         \
            const uint32_t ca = q6k_code<Q>(qa0, qa1, ha, u), cb = q6k_code<Q>(qb0, qb1, hb, u); \
            uint32_t A[4];                                                                      \
            A[0] = h2_fma(h_pair01(ca), s2a, b2a);                                              \
            A[1] = h2_fma(h_pair01(cb), s2b, b2b);                                              \
            A[2] = h2_fma(h_pair23(ca), s2a, b2a);                                              \
            A[3] = h2_fma(h_pair23(cb), s2b, b2b);                                              \
            mma_f16_16816(D, A, x[8 * (Q) + 2 * u], x[8 * (Q) + 2 * u + 1]);                    \
        }                                                                                       \
    }
    QMM_MVH_Q6K_QUAD(0)
    QMM_MVH_Q6K_QUAD(1)
    QMM_MVH_Q6K_QUAD(2)
    QMM_MVH_Q6K_QUAD(3)
#undef QMM_MVH_Q6K_QUAD
    return true;
}

// The same for any int8 scale: sc * (q - 32) as lo * (q - 32) + 8 hi * (q -
// 32), both exact in fp16, in two MMAs.
template <int QW>
__device__ __forceinline__ void q6k_tile_exact(uint32_t slot, int ra, int rb, int c, uint32_t sel,
                                            const uint32_t (&x)[32], float (&D)[4]) {
    uint32_t qa0[4], qa1[4], ha[4], sa[4], qb0[4], qb1[4], hb[4], sb[4];
    mvh_seg<QW>(slot, ra, c, sel, qa0);
    mvh_seg<QW>(slot, ra, 4 + c, sel, qa1);
    mvh_seg<QW>(slot, ra, 8 + c, sel, ha);
    mvh_seg<QW>(slot, ra, 12, sel, sa);
    mvh_seg<QW>(slot, rb, c, sel, qb0);
    mvh_seg<QW>(slot, rb, 4 + c, sel, qb1);
    mvh_seg<QW>(slot, rb, 8 + c, sel, hb);
    mvh_seg<QW>(slot, rb, 12, sel, sb);
#pragma unroll
    for (int Q = 0; Q < 4; ++Q) {
        const int s0 = q6k_sc(sa[Q], c), s1 = q6k_sc(sb[Q], c);
        const int l0 = s0 & 7, l1 = s1 & 7;
        const uint32_t lo_a = h2_splat(l0), lo_b = h2_splat(l1);
        const uint32_t hi_a = h2_splat(s0 - l0), hi_b = h2_splat(s1 - l1);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t ca, cb;
            if (Q == 0) { ca = q6k_code<0>(qa0, qa1, ha, u); cb = q6k_code<0>(qb0, qb1, hb, u); }
            else if (Q == 1) { ca = q6k_code<1>(qa0, qa1, ha, u); cb = q6k_code<1>(qb0, qb1, hb, u); }
            else if (Q == 2) { ca = q6k_code<2>(qa0, qa1, ha, u); cb = q6k_code<2>(qb0, qb1, hb, u); }
            else { ca = q6k_code<3>(qa0, qa1, ha, u); cb = q6k_code<3>(qb0, qb1, hb, u); }
            const uint32_t ea0 = h2_add(h_pair01(ca), kH2M1056), eb0 = h2_add(h_pair01(cb), kH2M1056);
            const uint32_t ea1 = h2_add(h_pair23(ca), kH2M1056), eb1 = h2_add(h_pair23(cb), kH2M1056);
            uint32_t A[4];
            A[0] = h2_mul(ea0, lo_a);
            A[1] = h2_mul(eb0, lo_b);
            A[2] = h2_mul(ea1, lo_a);
            A[3] = h2_mul(eb1, lo_b);
            mma_f16_16816(D, A, x[8 * Q + 2 * u], x[8 * Q + 2 * u + 1]);
            A[0] = h2_mul(ea0, hi_a);
            A[1] = h2_mul(eb0, hi_b);
            A[2] = h2_mul(ea1, hi_a);
            A[3] = h2_mul(eb1, hi_b);
            mma_f16_16816(D, A, x[8 * Q + 2 * u], x[8 * Q + 2 * u + 1]);
        }
    }
}

// One q6_K stage of both tiles of an item: acc[t] += d * (tile t's sum).
template <int QW>
__device__ __forceinline__ void q6k_stage(uint32_t slot, int g, int c, uint32_t L, uint32_t selc,
                                          const uint32_t (&x)[32], float (&acc)[2][4]) {
    const uint32_t sel = (L & 2u) ? 0x5432u : 0x3210u;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int ra = 16 * t + g, rb = ra + 8;
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (!q6k_tile_fast<QW>(slot, ra, rb, c, sel, selc, x, D)) q6k_tile_exact<QW>(slot, ra, rb, c, sel, x, D);
        // d at byte 208 + L: piece 13, byte L of it (16 + L into box 3)
        const float da = half_bits_to_float(lds_u16(q6k_piece(slot, ra, 13) + L));
        const float db = half_bits_to_float(lds_u16(q6k_piece(slot, rb, 13) + L));
        acc[t][0] = fmaf(da, D[0], acc[t][0]);
        acc[t][1] = fmaf(da, D[1], acc[t][1]);
        acc[t][2] = fmaf(db, D[2], acc[t][2]);
        acc[t][3] = fmaf(db, D[3], acc[t][3]);
    }
}

// ------------------------------------------------------------ Q4_0 / Q8_0 stages
// Block b of the stage; lane c's weights 8c .. 8c + 7 (MMA u = 0: 8c .. + 3,
// u = 1: 8c + 4 .. + 7), whose activations are x[4b .. 4b + 3].
// Q4_0 (18 B: d | qs[16]): weight e is nibble e / 16 of qs[e % 16], so the
// lane's codes are nibble c / 2 of qs[8 (c % 2) .. + 7].
template <int BLK>
__device__ __forceinline__ void q4_0_block(uint32_t slot, int ra, int rb, int c, const uint32_t (&x)[32],
                                           float (&acc)[4]) {
    constexpr uint32_t o = 18 * BLK + 2;          // qs of block BLK (o % 4 is 0 for odd BLK, 2 for even)
    constexpr bool AL = (o % 4) == 0;
    const uint32_t oq = o + 8u * static_cast<uint32_t>(c & 1);
    const uint32_t sh = 4u * static_cast<uint32_t>(c >> 1);
    const uint32_t a0 = (mvh_word<AL>(slot, ra, oq) >> sh) & 0x0F0F0F0Fu;
    const uint32_t a1 = (mvh_word<AL>(slot, ra, oq + 4) >> sh) & 0x0F0F0F0Fu;
    const uint32_t b0 = (mvh_word<AL>(slot, rb, oq) >> sh) & 0x0F0F0F0Fu;
    const uint32_t b1 = (mvh_word<AL>(slot, rb, oq + 4) >> sh) & 0x0F0F0F0Fu;
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t A[4];
    A[0] = h2_add(h_pair01(a0), kH2M1032);
    A[1] = h2_add(h_pair01(b0), kH2M1032);
    A[2] = h2_add(h_pair23(a0), kH2M1032);
    A[3] = h2_add(h_pair23(b0), kH2M1032);
    mma_f16_16816(D, A, x[4 * BLK], x[4 * BLK + 1]);
    A[0] = h2_add(h_pair01(a1), kH2M1032);
    A[1] = h2_add(h_pair01(b1), kH2M1032);
    A[2] = h2_add(h_pair23(a1), kH2M1032);
    A[3] = h2_add(h_pair23(b1), kH2M1032);
    mma_f16_16816(D, A, x[4 * BLK + 2], x[4 * BLK + 3]);
    const float da = mvh_half(slot, ra, 18 * BLK), db = mvh_half(slot, rb, 18 * BLK);
    acc[0] = fmaf(da, D[0], acc[0]);
    acc[1] = fmaf(da, D[1], acc[1]);
    acc[2] = fmaf(db, D[2], acc[2]);
    acc[3] = fmaf(db, D[3], acc[3]);
}

// Q8_0 (34 B: d | qs[32] int8), blocks at lead L (0 or 8); the lane's codes
// are qs[8c .. 8c + 7].
template <int BLK>
__device__ __forceinline__ void q8_0_block(uint32_t slot, int ra, int rb, int c, uint32_t L,
                                           const uint32_t (&x)[32], float (&acc)[4]) {
    constexpr uint32_t o = 34 * BLK + 2;          // o % 4 is 0 for odd BLK, 2 for even (L % 4 == 0)
    constexpr bool AL = (o % 4) == 0;
    const uint32_t oq = L + o + 8u * static_cast<uint32_t>(c);
    const uint32_t a0 = mvh_word<AL>(slot, ra, oq) ^ 0x80808080u;
    const uint32_t a1 = mvh_word<AL>(slot, ra, oq + 4) ^ 0x80808080u;
    const uint32_t b0 = mvh_word<AL>(slot, rb, oq) ^ 0x80808080u;
    const uint32_t b1 = mvh_word<AL>(slot, rb, oq + 4) ^ 0x80808080u;
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t A[4];
    A[0] = h2_add(h_pair01(a0), kH2M1152);
    A[1] = h2_add(h_pair01(b0), kH2M1152);
    A[2] = h2_add(h_pair23(a0), kH2M1152);
    A[3] = h2_add(h_pair23(b0), kH2M1152);
    mma_f16_16816(D, A, x[4 * BLK], x[4 * BLK + 1]);
    A[0] = h2_add(h_pair01(a1), kH2M1152);
    A[1] = h2_add(h_pair01(b1), kH2M1152);
    A[2] = h2_add(h_pair23(a1), kH2M1152);
    A[3] = h2_add(h_pair23(b1), kH2M1152);
    mma_f16_16816(D, A, x[4 * BLK + 2], x[4 * BLK + 3]);
    const float da = mvh_half(slot, ra, L + 34 * BLK), db = mvh_half(slot, rb, L + 34 * BLK);
    acc[0] = fmaf(da, D[0], acc[0]);
    acc[1] = fmaf(da, D[1], acc[1]);
    acc[2] = fmaf(db, D[2], acc[2]);
    acc[3] = fmaf(db, D[3], acc[3]);
}

__device__ __forceinline__ void q4_0_stage(uint32_t slot, int g, int c, const uint32_t (&x)[32],
                                           float (&acc)[2][4]) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int ra = 16 * t + g, rb = ra + 8;
        q4_0_block<0>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<1>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<2>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<3>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<4>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<5>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<6>(slot, ra, rb, c, x, acc[t]);
        q4_0_block<7>(slot, ra, rb, c, x, acc[t]);
    }
}

__device__ __forceinline__ void q8_0_stage(uint32_t slot, int g, int c, uint32_t L, const uint32_t (&x)[32],
                                           float (&acc)[2][4]) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int ra = 16 * t + g, rb = ra + 8;
        q8_0_block<0>(slot, ra, rb, c, L, x, acc[t]);
        q8_0_block<1>(slot, ra, rb, c, L, x, acc[t]);
        q8_0_block<2>(slot, ra, rb, c, L, x, acc[t]);
        q8_0_block<3>(slot, ra, rb, c, L, x, acc[t]);
    }
}

// ------------------------------------------------------------ the kernel

__host__ __device__ constexpr int mvh_stage_k(int fmt) { return fmt == FMT_Q8_0 ? 128 : 256; }
__host__ __device__ constexpr int mvh_stage_bytes(int fmt) {
    return fmt == FMT_Q6_K ? 210 : (fmt == FMT_Q4_0 ? 144 : 136);
}

struct MvhCursor {
    int it, p, m;  // item, stage of the item, matrix
};

__device__ __forceinline__ void mvh_advance(const MvhGroup& g, int ks, int member, int nteams, MvhCursor& c) {
    c.p += ks;
    if (c.p < g.m[c.m].stages) return;
    c.p = member;
    c.it += nteams;
    while (c.m + 1 < g.nmat && c.it >= g.m[c.m + 1].item0) ++c.m;
}

// byte offset of stage p of row j (of every group) in a view row of W, and
// the stage's lead in its first 16-byte piece
__device__ __forceinline__ int64_t mvh_stage_off(const MvhMat& a, int j, int p) {
    return static_cast<int64_t>(j) * a.rowbytes + static_cast<int64_t>(p) * mvh_stage_bytes(a.fmt);
}

// Issues the TMA copies of the stage at cursor c into `slot` (completing on
// bar): lane k issues box k, from the 16-byte boundary at or below the
// stage's first byte.
__device__ __forceinline__ void mvh_issue(const MvhGroup& g, const MvhCursor& c, uint32_t slot, uint32_t bar,
                                          int lane) {
    const MvhMat& a = g.m[c.m];
    const int li = c.it - a.item0;
    const int j = li & 7, G0 = (li >> 3) * kMvhRows;
    const int nb = mvh_boxes(a.fmt);
    const uint32_t bw = mvh_box_w(a.fmt);
    const int64_t off = mvh_stage_off(a, j, c.p) & ~static_cast<int64_t>(15);
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb) * bw * kMvhRows);
    __syncwarp();
    if (lane < nb)
        tma_load_2d(slot + static_cast<uint32_t>(lane) * bw * kMvhRows, &g.map[c.m],
                    static_cast<int>(off / 2) + static_cast<int>(bw / 2) * lane, G0, bar);
}

// The lane's activations of stage p of matrix a (batch row g; zero past B).
__device__ __forceinline__ void mvh_x_fetch(const MvhGroup& g, const MvhMat& a, int p, int lane,
                                            uint32_t (&x)[32]) {
    const int gr = lane >> 2, c = lane & 3;
    if (gr < g.B) {
        const int64_t k0 = static_cast<int64_t>(p) * mvh_stage_k(a.fmt);
        const __half* xr = reinterpret_cast<const __half*>(a.xh) + static_cast<int64_t>(gr) * a.K + k0;
        if (a.fmt == FMT_Q6_K) {
#pragma unroll
            for (int Q = 0; Q < 4; ++Q) {
                const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * (c + 4 * Q)));
                const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * (c + 4 * Q) + 8));
                x[8 * Q + 0] = v0.x; x[8 * Q + 1] = v0.y; x[8 * Q + 2] = v0.z; x[8 * Q + 3] = v0.w;
                x[8 * Q + 4] = v1.x; x[8 * Q + 5] = v1.y; x[8 * Q + 6] = v1.z; x[8 * Q + 7] = v1.w;
            }
        } else {
            const int nb = mvh_stage_k(a.fmt) / 32;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (b < nb) v = __ldg(reinterpret_cast<const uint4*>(xr + 32 * b + 8 * c));
                x[4 * b + 0] = v.x; x[4 * b + 1] = v.y; x[4 * b + 2] = v.z; x[4 * b + 3] = v.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0u;
    }
}

// Bounded wait for the TMA copies of a slot; false (and the error word set)
// after the time limit.
__device__ __forceinline__ bool mvh_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((it & 15u) == 0) {
            int late = globaltimer_ns() - t0 > kWaitLimitNs ? 1 : 0;
            late = __shfl_sync(0xffffffffu, late, 0);
            if (late) {
                if ((threadIdx.x & 31) == 0) atomicOr(err, DERR_GEMV_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mvh_team_sync(int team, int ks) {
    if (ks > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * ks) : "memory");
}

__global__ void __launch_bounds__(kMvhWarps * 32, 1) mvh_kernel(const __grid_constant__ MvhGroup g) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, c = lane & 3;
    const int ks = g.ks;
    const int team = warp / ks, member = warp % ks;
    const uint32_t S = smem_u32(smem);
    const uint32_t ring = S + static_cast<uint32_t>(warp) * kMvhNS * kMvhSlot;
    const uint32_t bars = S + kMvhBarOff + static_cast<uint32_t>(warp) * kMvhNS * 8;
    float* part = reinterpret_cast<float*>(smem + kMvhPartOff);
    const int nteams = static_cast<int>(gridDim.x) * (kMvhWarps / ks);
    const int gt = team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    // byte selector: byte c of a word into the low bytes of two fp16 (1024 + byte)
    const uint32_t selc = 0x4040u | (static_cast<uint32_t>(c) << 8) | static_cast<uint32_t>(c);

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (gt >= g.items) return;  // the whole team: every member has the same items
    if (lane < kMvhNS) mbar_init(bars + 8 * lane, 1);
    fence_mbar_init();
    __syncwarp();

    // the weights do not depend on the previous kernel: the first copies go
    // out before waiting for it
    MvhCursor ic{gt, member, 0};
    while (ic.m + 1 < g.nmat && ic.it >= g.m[ic.m + 1].item0) ++ic.m;
    const int m0 = ic.m;
    uint32_t issued = 0, used = 0;
    for (int j = 0; j < kMvhNS - 1 && ic.it < g.items; ++j) {
        mvh_issue(g, ic, ring + (issued % kMvhNS) * kMvhSlot, bars + 8 * (issued % kMvhNS), lane);
        ++issued;
        mvh_advance(g, ks, member, nteams, ic);
    }
    grid_dependency_wait();  // x comes from the prep kernel

    bool ok = true;
    uint32_t x[32], xn[32];
    mvh_x_fetch(g, g.m[m0], member, lane, xn);
    int m = m0;
    for (int it = gt; it < g.items; it += nteams) {
        while (m + 1 < g.nmat && it >= g.m[m + 1].item0) ++m;
        const MvhMat& a = g.m[m];
        const int li = it - a.item0;
        const int j = li & 7, G0 = (li >> 3) * kMvhRows;
        float acc[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[t][q] = 0.0f;
        for (int p = member; p < a.stages; p += ks) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = xn[i];
            // the next stage's activations (this item's, or the next item's first)
            if (p + ks < a.stages) {
                mvh_x_fetch(g, a, p + ks, lane, xn);
            } else if (it + nteams < g.items) {
                int mn = m;
                while (mn + 1 < g.nmat && it + nteams >= g.m[mn + 1].item0) ++mn;
                mvh_x_fetch(g, g.m[mn], member, lane, xn);
            }
            // the copies NS - 1 stages ahead, into the slot consumed last
            if (ic.it < g.items) {
                fence_proxy_async_smem();
                __syncwarp();
                mvh_issue(g, ic, ring + (issued % kMvhNS) * kMvhSlot, bars + 8 * (issued % kMvhNS), lane);
                ++issued;
                mvh_advance(g, ks, member, nteams, ic);
            }
            const uint32_t slot = ring + (used % kMvhNS) * kMvhSlot;
            if (ok) ok = mvh_wait(bars + 8 * (used % kMvhNS), (used / kMvhNS) & 1u, g.st.err);
            ++used;
            const uint32_t L = static_cast<uint32_t>(mvh_stage_off(a, j, p) & 15);
            if (a.fmt == FMT_Q6_K) {
                switch (L >> 2) {
                    case 0: q6k_stage<0>(slot, gr, c, L, selc, x, acc); break;
                    case 1: q6k_stage<1>(slot, gr, c, L, selc, x, acc); break;
                    case 2: q6k_stage<2>(slot, gr, c, L, selc, x, acc); break;
                    default: q6k_stage<3>(slot, gr, c, L, selc, x, acc); break;
                }
            } else if (a.fmt == FMT_Q4_0) {
                q4_0_stage(slot, gr, c, x, acc);
            } else {
                q8_0_stage(slot, gr, c, L, x, acc);
            }
            __syncwarp();
        }
        // the team's sums of the item, added by member 0 in member order
        if (ks > 1) {
#pragma unroll
            for (int q = 0; q < 8; ++q) part[(warp * 8 + q) * 32 + lane] = acc[q >> 2][q & 3];
            mvh_team_sync(team, ks);
            if (member == 0) {
                for (int t2 = 1; t2 < ks; ++t2)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q >> 2][q & 3] += part[((warp + t2) * 8 + q) * 32 + lane];
            }
            mvh_team_sync(team, ks);  // the partial sums are read before they are overwritten
        }
        if (member == 0) {
            // lane (g, c): item rows 16t + g and 16t + g + 8, batch rows 2c, 2c + 1
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
                const int b = 2 * c + b2;
                if (b >= g.B) continue;
                const float sc = a.xinv[b];
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int64_t n = static_cast<int64_t>(j) + 8 * (G0 + 16 * t + gr + 8 * h);
                        if (n < a.N) a.y[static_cast<int64_t>(b) * a.N + n] = acc[t][2 * h + b2] * sc;
                    }
            }
        }
    }
    // a slot whose wait gave up may still be receiving: wait for it (bounded)
    // before the CTA's shared memory is released
    if (!ok)
        for (uint32_t u = used > kMvhNS ? used - kMvhNS : 0; u < issued; ++u)
            (void)mvh_wait(bars + 8 * (u % kMvhNS), (u / kMvhNS) & 1u, g.st.err);
}

}  // namespace qmm
