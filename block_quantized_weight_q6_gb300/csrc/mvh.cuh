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
// Work item: 16 rows of one matrix at stride 8 (rows j + 8 (G + i), i < 16),
// all of K in stages (q6_K one super-block, Q4_0 8 blocks, Q8_0 4 blocks).
// Rows 8 apart start at the same offset modulo 16 (the pitch of 8 rows is a
// multiple of 16 for every even row size), so the byte lead of a stage is
// the same for all 16 rows of an item and the realignment of the code bytes
// is warp-uniform. A stage arrives by 2-D TMA with W seen as
// [N / 8][8 * rowbytes] 16-bit elements, in boxes 16 rows high that land
// row after row: q6_K four boxes 64 bytes wide (the 14 pieces of 16 bytes a
// super-block and its lead cover, and 2 more), so the 128-bit loads of one
// load phase (rows 2k and 2k + 1, lanes c = 0..3 reading pieces c + s) hit 32
// different banks; Q4_0 / Q8_0 one box 144 bytes wide (their stage, lead
// included), read with 32- and 64-bit loads at a row base plus a constant. Box
// destinations are 128-byte aligned.
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
constexpr int kMvhRows = 16;                // rows per item: one 16-row MMA tile
// box width in bytes and boxes per stage: q6_K 4 x 64, Q4_0 / Q8_0 / Q4_K
// 1 x 144, Q2_K 1 x 96 (its 84-byte super-block and a lead of up to 12)
__host__ __device__ constexpr uint32_t mvh_box_w(int fmt) {
    return fmt == FMT_Q6_K ? 64u : (fmt == FMT_Q2_K ? 96u : 144u);
}
__host__ __device__ constexpr int mvh_boxes(int fmt) { return fmt == FMT_Q6_K ? 4 : 1; }
constexpr uint32_t kMvhRow32 = 144;  // Q4_0 / Q8_0 / Q4_K row stride in a stage slot
constexpr uint32_t kMvhRowQ2K = 96;  // Q2_K row stride in a stage slot
constexpr uint32_t kMvhSlot = 4 * 64 * kMvhRows;   // the largest stage: 4 KB
constexpr uint32_t kMvhPartOff = kMvhWarps * kMvhNS * kMvhSlot;  // team sums, after the rings
constexpr uint32_t kMvhBarOff = kMvhPartOff + kMvhWarps * 4 * 32 * 4;
constexpr uint32_t kMvhFifoOff = kMvhBarOff + kMvhWarps * kMvhNS * 8;  // per warp: 4 item numbers
constexpr uint32_t kMvhSmem = kMvhFifoOff + kMvhWarps * 16;
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
constexpr uint32_t kH2One = 0x3C003C00u;       // (1, 1)
constexpr uint32_t kH2Sixteenth = 0x2C002C00u; // (1/16, 1/16)
constexpr uint32_t kH2M72 = 0xD480D480u;       // (-72, -72): (1024 + 16 q) / 16 - 72 = q - 8
constexpr uint32_t kH2M1024 = 0xE400E400u;     // (-1024, -1024)
constexpr uint32_t kH2Quarter = 0x34003400u;   // (1/4, 1/4)
constexpr uint32_t kH2Sixtyfourth = 0x24002400u;  // (1/64, 1/64)
constexpr uint32_t kH2M256 = 0xDC00DC00u;      // -1024 / 4
constexpr uint32_t kH2M64 = 0xD400D400u;       // -1024 / 16
constexpr uint32_t kH2M16 = 0xCC00CC00u;       // -1024 / 64

__device__ __forceinline__ void mvh_lds_v4(uint32_t a, uint32_t* w) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(a));
}

// q6_K stage slot: offset of 16-byte piece p of a row from the row's base
// (slot + 64 r): four boxes of [kMvhRows rows][64 B].
__host__ __device__ constexpr uint32_t q6k_poff(int p) {
    return static_cast<uint32_t>(p >> 2) * (64u * kMvhRows) + 16u * static_cast<uint32_t>(p & 3);
}

// The lane's piece offsets (pieces c, c + 1, 4 + c, 5 + c, 8 + c, 9 + c),
// computed once.
struct Q6Off {
    uint32_t o[6];
};

// The 16 bytes at byte lead L (even, < 16; QW = L / 4 and sel shifts by
// L % 4) of the pieces at row base + oa and row base + ob.
template <int QW>
__device__ __forceinline__ void mvh_seg(uint32_t row, uint32_t oa, uint32_t ob, uint32_t sel, uint32_t (&o)[4]) {
    uint32_t w[8];
    mvh_lds_v4(row + oa, w);
    mvh_lds_v4(row + ob, w + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __byte_perm(w[QW + i], w[QW + i + 1], sel);
}

// The scale segment (16 bytes at lead L of pieces 12, 13) and the
// super-block's d, which follows it (bytes 208, 209 of the super-block).
template <int QW>
__device__ __forceinline__ uint32_t mvh_seg_sc_d(uint32_t row, uint32_t sel, uint32_t L, uint32_t (&o)[4]) {
    uint32_t w[8];
    mvh_lds_v4(row + q6k_poff(12), w);
    mvh_lds_v4(row + q6k_poff(13), w + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __byte_perm(w[QW + i], w[QW + i + 1], sel);
    return (w[4 + QW] >> (8u * (L & 2u))) & 0xFFFFu;
}

// Q4_0 / Q8_0: four bytes at offset o (a compile-time constant) from the
// lane's row base; ALIGNED says whether the base + o is a multiple of 4
// (else it is 2 past one, and the word is put together from the aligned
// words around it).
template <bool ALIGNED, uint32_t O>
__device__ __forceinline__ uint32_t mvh_word(uint32_t base) {
    if constexpr (ALIGNED) {
        return lds_u32(base + O);
    } else {
        return __byte_perm(lds_u32(base + O - 2), lds_u32(base + O + 2), 0x5432);
    }
}

// Eight activations (16 bytes) at element offset off of the lane's row xr.
// (A lane past the batch reads a valid row too: its MMA column is never
// stored, so no load needs a predicate.)
__device__ __forceinline__ uint4 mvh_x8(const uint16_t* xr, int off) {
    return __ldg(reinterpret_cast<const uint4*>(xr + off));
}

// ------------------------------------------------------------ q6_K stage
// The 16-row tile: rows g and g + 8 of the stage for lane (g, c). Lane c's
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

// The tile's sum over one super-block: sc * (q - 32) from (1024 + c) * sc -
// 1056 * sc in one fp16 FMA, exact for |sc| <= 62. A scale outside that range
// makes the bias -1056 * sc overflow to an infinity, so the sum is not finite
// and the caller recomputes the tile in the exact form. Four accumulator
// chains (one per position u in the group) keep consecutive MMAs independent.
// pa, pb: the bases (slot + 64 r) of the tile's rows g and g + 8.
template <int QW>
__device__ __forceinline__ float4 q6k_tile_fast(uint32_t pa, uint32_t pb, const Q6Off& po, uint32_t sel, uint32_t L,
                                                uint32_t selc, const uint16_t* xr, int c, float& da, float& db) {
    uint32_t qa0[4], qa1[4], ha[4], sa[4], qb0[4], qb1[4], hb[4], sb[4];
    da = half_bits_to_float(mvh_seg_sc_d<QW>(pa, sel, L, sa));
    db = half_bits_to_float(mvh_seg_sc_d<QW>(pb, sel, L, sb));
    mvh_seg<QW>(pa, po.o[0], po.o[1], sel, qa0);
    mvh_seg<QW>(pb, po.o[0], po.o[1], sel, qb0);
    mvh_seg<QW>(pa, po.o[4], po.o[5], sel, ha);
    mvh_seg<QW>(pb, po.o[4], po.o[5], sel, hb);
    // one accumulator per u: the four MMAs of a quad are independent
    float D[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) D[u][q] = 0.0f;
#define QMM_MVH_Q6K_QUAD(Q)                                                                          \
    {                                                                                                \
        const uint4 x0 = mvh_x8(xr, 16 * (c + 4 * (Q))), x1 = mvh_x8(xr, 16 * (c + 4 * (Q)) + 8);    \
        const uint32_t xq[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};                   \
        const uint32_t s2a = h2_add(__byte_perm(sa[Q] ^ 0x80808080u, 0x64646464u, selc), kH2M1152);   \
        const uint32_t s2b = h2_add(__byte_perm(sb[Q] ^ 0x80808080u, 0x64646464u, selc), kH2M1152);   \
        const uint32_t b2a = h2_mul(s2a, kH2M1056), b2b = h2_mul(s2b, kH2M1056);                     \
        _Pragma("unroll") for (int u = 0; u < 4; ++u) {                                              \
            const uint32_t ca = q6k_code<Q>(qa0, qa1, ha, u), cb = q6k_code<Q>(qb0, qb1, hb, u);      \
            uint32_t A[4];                                                                           \
            A[0] = h2_fma(h_pair01(ca), s2a, b2a);                                                   \
            A[1] = h2_fma(h_pair01(cb), s2b, b2b);                                                   \
            A[2] = h2_fma(h_pair23(ca), s2a, b2a);                                                   \
            A[3] = h2_fma(h_pair23(cb), s2b, b2b);                                                   \
            mma_f16_16816(D[u], A, xq[2 * u], xq[2 * u + 1]);                                        \
        }                                                                                            \
    }
    // the low-nibble quads of ql 16c.. (Q = 0, 2) first, then ql 64 + 16c.. (Q = 1, 3)
    QMM_MVH_Q6K_QUAD(0)
    QMM_MVH_Q6K_QUAD(2)
    mvh_seg<QW>(pa, po.o[2], po.o[3], sel, qa1);
    mvh_seg<QW>(pb, po.o[2], po.o[3], sel, qb1);
    QMM_MVH_Q6K_QUAD(1)
    QMM_MVH_Q6K_QUAD(3)
#undef QMM_MVH_Q6K_QUAD
    return make_float4((D[0][0] + D[1][0]) + (D[2][0] + D[3][0]), (D[0][1] + D[1][1]) + (D[2][1] + D[3][1]),
                       (D[0][2] + D[1][2]) + (D[2][2] + D[3][2]), (D[0][3] + D[1][3]) + (D[2][3] + D[3][3]));
}

// The same tile sum for any int8 scale, as lo * (q - 32) + 8 hi * (q - 32)
// (sc = lo + 8 hi, 0 <= lo < 8), both exact in fp16, in two MMAs. Kept out
// of line (it only runs for scales outside -62..62): it reads the code bytes
// byte by byte and the activations itself.
__device__ __noinline__ float4 q6k_tile_exact(uint32_t pa, uint32_t pb, int c, uint32_t L, const uint16_t* xrow) {
    uint32_t seg[2][4][4];  // row, segment (ql c, ql 4 + c, qh c, scales), word
    const uint32_t rows[2] = {pa, pb};
    const int piece[4] = {c, 4 + c, 8 + c, 12};
    for (int r = 0; r < 2; ++r)
        for (int q = 0; q < 4; ++q)
            for (int i = 0; i < 4; ++i) {
                uint32_t w = 0;
                for (int bt = 0; bt < 4; ++bt) {
                    const uint32_t o = L + 4 * i + bt;  // byte inside the piece pair
                    const uint32_t v =
                        lds_u16(rows[r] + q6k_poff(piece[q] + static_cast<int>(o >> 4)) + ((o & 15u) & ~1u));
                    w |= ((v >> (8 * (o & 1u))) & 0xFFu) << (8 * bt);
                }
                seg[r][q][i] = w;
            }
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int Q = 0; Q < 4; ++Q) {
        uint32_t lo2[2], hi2[2];
        for (int r = 0; r < 2; ++r) {
            const int sc = q6k_sc(seg[r][3][Q], c);
            lo2[r] = h2_splat(sc & 7);
            hi2[r] = h2_splat(sc - (sc & 7));
        }
        for (int u = 0; u < 4; ++u) {
            uint32_t cw[2];
            for (int r = 0; r < 2; ++r) {
                const uint32_t l = seg[r][Q & 1][u];
                const uint32_t lo = (Q >> 1) ? (l >> 4) : l;
                const uint32_t hi = ((seg[r][2][u] >> (2 * Q)) & 0x03030303u) << 4;
                cw[r] = (lo & 0x0F0F0F0Fu) | hi;
            }
            const uint32_t* xs = reinterpret_cast<const uint32_t*>(xrow + 16 * (c + 4 * Q) + 4 * u);
            const uint32_t b0 = xs[0], b1 = xs[1];
            const uint32_t e[4] = {h2_add(h_pair01(cw[0]), kH2M1056), h2_add(h_pair01(cw[1]), kH2M1056),
                                   h2_add(h_pair23(cw[0]), kH2M1056), h2_add(h_pair23(cw[1]), kH2M1056)};
            uint32_t A[4] = {h2_mul(e[0], lo2[0]), h2_mul(e[1], lo2[1]), h2_mul(e[2], lo2[0]),
                             h2_mul(e[3], lo2[1])};
            mma_f16_16816(D, A, b0, b1);
            const uint32_t Ah[4] = {h2_mul(e[0], hi2[0]), h2_mul(e[1], hi2[1]), h2_mul(e[2], hi2[0]),
                                    h2_mul(e[3], hi2[1])};
            mma_f16_16816(D, Ah, b0, b1);
        }
    }
    return make_float4(D[0], D[1], D[2], D[3]);
}

__device__ __forceinline__ bool f4_finite(float4 v) {
    return isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w);
}

// One q6_K stage of the item's tile: acc += d * (the tile's sum).
// xr: the lane's activation row at the stage's first K.
__device__ __forceinline__ void q6k_stage(uint32_t slot, int g, int c, const Q6Off& po, uint32_t L, uint32_t selc,
                                          const uint16_t* xr, float (&acc)[4]) {
    const uint32_t sel = (L & 2u) ? 0x5432u : 0x3210u;
    const uint32_t pa = slot + 64u * static_cast<uint32_t>(g), pb = pa + 64u * 8u;
    float4 D;
    float da, db;
    switch (L >> 2) {
        case 0: D = q6k_tile_fast<0>(pa, pb, po, sel, L, selc, xr, c, da, db); break;
        case 1: D = q6k_tile_fast<1>(pa, pb, po, sel, L, selc, xr, c, da, db); break;
        case 2: D = q6k_tile_fast<2>(pa, pb, po, sel, L, selc, xr, c, da, db); break;
        default: D = q6k_tile_fast<3>(pa, pb, po, sel, L, selc, xr, c, da, db); break;
    }
    if (__any_sync(0xffffffffu, !f4_finite(D))) D = q6k_tile_exact(pa, pb, c, L, xr);
    acc[0] = fmaf(da, D.x, acc[0]);
    acc[1] = fmaf(da, D.y, acc[1]);
    acc[2] = fmaf(db, D.z, acc[2]);
    acc[3] = fmaf(db, D.w, acc[3]);
}

// ------------------------------------------------------------ Q4_0 / Q8_0 stages
// Block BLK of the stage; lane c's weights 8c .. 8c + 7 (MMA u = 0: 8c .. + 3,
// u = 1: 8c + 4 .. + 7). Rows are 144 bytes apart in the slot.

// two consecutive 32-bit words at an 8-byte-aligned shared address
__device__ __forceinline__ void mvh_lds_v2(uint32_t a, uint32_t& w0, uint32_t& w1) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(a));
}

// The lane's eight code bytes at base + O (base a multiple of 8, O even), each
// masked with m (FLIP: with the top bit flipped instead), as four fp16 pairs
// p[i] = (1024 + byte 2i, 1024 + byte 2i + 1). Both steps are bytewise, so
// they work on the aligned words around the bytes: for O % 4 == 2 the pairs
// are the upper half of one word and the lower half of the next, and no word
// is put together first.
template <bool FLIP>
__device__ __forceinline__ uint32_t mvh_code_word(uint32_t w, uint32_t m) {
    return FLIP ? (w ^ 0x80808080u) : (w & m);
}

template <uint32_t O, bool FLIP>
__device__ __forceinline__ void mvh_code_pairs(uint32_t base, uint32_t m, uint32_t (&p)[4]) {
    if constexpr (O % 4 == 0) {
        uint32_t w0, w1;
        if constexpr (O % 8 == 0) {
            mvh_lds_v2(base + O, w0, w1);
        } else {
            w0 = lds_u32(base + O);
            w1 = lds_u32(base + O + 4);
        }
        w0 = mvh_code_word<FLIP>(w0, m);
        w1 = mvh_code_word<FLIP>(w1, m);
        p[0] = h_pair01(w0);
        p[1] = h_pair23(w0);
        p[2] = h_pair01(w1);
        p[3] = h_pair23(w1);
    } else {
        uint32_t lo, mid, hi;
        if constexpr ((O - 2) % 8 == 0) {
            mvh_lds_v2(base + O - 2, lo, mid);
        } else {
            lo = lds_u32(base + O - 2);
            mid = lds_u32(base + O + 2);
        }
        hi = lds_u32(base + O + 6);
        lo = mvh_code_word<FLIP>(lo, m);
        mid = mvh_code_word<FLIP>(mid, m);
        hi = mvh_code_word<FLIP>(hi, m);
        p[0] = h_pair23(lo);
        p[1] = h_pair01(mid);
        p[2] = h_pair23(mid);
        p[3] = h_pair01(hi);
    }
}

// The two MMAs of a block from the code pairs of rows g (pa) and g + 8 (pb):
// A = pair * hm + ha, the lane's signed codes, exact in fp16.
__device__ __forceinline__ void mvh_block_mma(const uint32_t (&pa)[4], const uint32_t (&pb)[4], uint32_t hm,
                                              uint32_t ha, uint4 xv, float (&D)[4]) {
    uint32_t A[4];
    A[0] = h2_fma(pa[0], hm, ha);
    A[1] = h2_fma(pb[0], hm, ha);
    A[2] = h2_fma(pa[1], hm, ha);
    A[3] = h2_fma(pb[1], hm, ha);
    mma_f16_16816(D, A, xv.x, xv.y);
    A[0] = h2_fma(pa[2], hm, ha);
    A[1] = h2_fma(pb[2], hm, ha);
    A[2] = h2_fma(pa[3], hm, ha);
    A[3] = h2_fma(pb[3], hm, ha);
    mma_f16_16816(D, A, xv.z, xv.w);
}

// Q4_0 (18 B: d | qs[16]), lead 0: weight e is nibble e / 16 of qs[e % 16],
// so the lane's codes are nibble c / 2 of qs[8 (c % 2) .. + 7]. The nibble is
// masked in place: a low nibble q gives the pair value 1024 + q, a high one
// 1024 + 16 q, and A = (1024 + q) - 1032 or (1024 + 16 q) / 16 - 72, both
// q - 8. ra, rb: the rows' bases (slot + 144 r); la, lb: the same plus
// 8 (c % 2); nm, hm, ha: the lane's nibble mask, multiplier and addend.
template <int BLK>
__device__ __forceinline__ void q4_0_block(uint32_t ra, uint32_t rb, uint32_t la, uint32_t lb, uint32_t nm,
                                           uint32_t hm, uint32_t ha, int c, const uint16_t* xr, float (&acc)[4]) {
    constexpr uint32_t O = 18 * BLK + 2;  // qs of block BLK: O % 4 is 0 for odd BLK, 2 for even
    const uint4 xv = mvh_x8(xr, 32 * BLK + 8 * c);
    uint32_t pa[4], pb[4];
    mvh_code_pairs<O, false>(la, nm, pa);
    mvh_code_pairs<O, false>(lb, nm, pb);
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mvh_block_mma(pa, pb, hm, ha, xv, D);
    const float da = half_bits_to_float(lds_u16(ra + 18 * BLK)), db = half_bits_to_float(lds_u16(rb + 18 * BLK));
    acc[0] = fmaf(da, D[0], acc[0]);
    acc[1] = fmaf(da, D[1], acc[1]);
    acc[2] = fmaf(db, D[2], acc[2]);
    acc[3] = fmaf(db, D[3], acc[3]);
}

// Q8_0 (34 B: d | qs[32] int8), blocks at lead L (0 or 8); the lane's codes
// are qs[8c .. 8c + 7], flipped to v ^ 128 = v + 128, so A = (1024 + (v ^
// 128)) - 1152 = v. ra, rb: the rows' bases plus L; la, lb: plus 8c more.
template <int BLK>
__device__ __forceinline__ void q8_0_block(uint32_t ra, uint32_t rb, uint32_t la, uint32_t lb, int c,
                                           const uint16_t* xr, float (&acc)[4]) {
    constexpr uint32_t O = 34 * BLK + 2;  // O % 4 is 0 for odd BLK, 2 for even (L % 8 == 0)
    const uint4 xv = mvh_x8(xr, 32 * BLK + 8 * c);
    uint32_t pa[4], pb[4];
    mvh_code_pairs<O, true>(la, 0u, pa);
    mvh_code_pairs<O, true>(lb, 0u, pb);
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mvh_block_mma(pa, pb, kH2One, kH2M1152, xv, D);
    const float da = half_bits_to_float(lds_u16(ra + 34 * BLK)), db = half_bits_to_float(lds_u16(rb + 34 * BLK));
    acc[0] = fmaf(da, D[0], acc[0]);
    acc[1] = fmaf(da, D[1], acc[1]);
    acc[2] = fmaf(db, D[2], acc[2]);
    acc[3] = fmaf(db, D[3], acc[3]);
}

__device__ __forceinline__ void q4_0_stage(uint32_t slot, int g, int c, const uint16_t* xr, float (&acc)[4]) {
    const bool high = (c >> 1) != 0;
    const uint32_t nm = high ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    const uint32_t hm = high ? kH2Sixteenth : kH2One, ha = high ? kH2M72 : kH2M1032;
    const uint32_t lo = 8u * static_cast<uint32_t>(c & 1);
    const uint32_t ra = slot + kMvhRow32 * static_cast<uint32_t>(g), rb = ra + 8u * kMvhRow32;
    const uint32_t la = ra + lo, lb = rb + lo;
    q4_0_block<0>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<1>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<2>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<3>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<4>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<5>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<6>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
    q4_0_block<7>(ra, rb, la, lb, nm, hm, ha, c, xr, acc);
}

__device__ __forceinline__ void q8_0_stage(uint32_t slot, int g, int c, uint32_t L, const uint16_t* xr,
                                           float (&acc)[4]) {
    const uint32_t ra = slot + kMvhRow32 * static_cast<uint32_t>(g) + L, rb = ra + 8u * kMvhRow32;
    const uint32_t la = ra + 8u * static_cast<uint32_t>(c), lb = rb + 8u * static_cast<uint32_t>(c);
    q8_0_block<0>(ra, rb, la, lb, c, xr, acc);
    q8_0_block<1>(ra, rb, la, lb, c, xr, acc);
    q8_0_block<2>(ra, rb, la, lb, c, xr, acc);
    q8_0_block<3>(ra, rb, la, lb, c, xr, acc);
}

// ------------------------------------------------------------ Q4_K / Q2_K stages
// The K-quant ladder formats (quantprobe "LAWS.md", Law 4 amendment L-16):
// weight = d * sc_j * q - dmin * m_j per sub-block j. A = sc_j * q is exact
// in fp16 (<= 63 * 15), made like Q4_0's from the code masked in place by
// one fp16x2 FMA per pair, with the sub-block's scale folded into the FMA's
// multiplier and addend. The min term is a second MMA on the same
// activations with A = m_j (exact), so a stage keeps two sums per row, D1 =
// sum sc q x and D2 = sum m x, and adds d D1 - dmin D2 once per super-block.
// Lane c takes sub-blocks c + 4t of its two rows, so the scales and mins it
// needs are its own: four consecutive weights of a sub-block per MMA.

// (1024 + byte c of w) in both halves; selc = 0x4040 | c << 8 | c
__device__ __forceinline__ uint32_t h_byte_pair(uint32_t w, uint32_t selc) {
    return __byte_perm(w, 0x64646464u, selc);
}

// FMA operands of a sub-block: A = pair * hm + ha (hm = sc * f, ha = -1024 hm,
// f undoing the code's place in its byte), and the min pair for D2
struct KqSub {
    uint32_t hm, ha, m;
};

// from the sub-block's scale and min bytes (byte c of sc4 / m4, each < 64)
__device__ __forceinline__ KqSub kq_sub(uint32_t sc4, uint32_t m4, uint32_t selc, uint32_t f, uint32_t nf) {
    KqSub o;
    o.hm = h2_fma(h_byte_pair(sc4, selc), f, nf);  // (1024 + sc) f - 1024 f = sc f, exact
    o.ha = h2_mul(o.hm, kH2M1024);
    o.m = h2_add(h_byte_pair(m4, selc), kH2M1024);
    return o;
}

// the four MMAs of one code word quad (words w[0..3] of both rows, masked
// with nm): word u holds weights 4u .. 4u + 3, whose activations are x[4u ..]
__device__ __forceinline__ void kq_mma4(const uint32_t (&wa)[4], const uint32_t (&wb)[4], uint32_t nm,
                                        const KqSub& sa, const KqSub& sb, uint4 x0, uint4 x1, float (&D1)[4],
                                        float (&D2)[4]) {
    const uint32_t A2[4] = {sa.m, sb.m, sa.m, sb.m};
    const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t a = wa[u] & nm, b = wb[u] & nm;
        uint32_t A[4];
        A[0] = h2_fma(h_pair01(a), sa.hm, sa.ha);
        A[1] = h2_fma(h_pair01(b), sb.hm, sb.ha);
        A[2] = h2_fma(h_pair23(a), sa.hm, sa.ha);
        A[3] = h2_fma(h_pair23(b), sb.hm, sb.ha);
        mma_f16_16816(D1, A, xb[2 * u], xb[2 * u + 1]);
        mma_f16_16816(D2, A2, xb[2 * u], xb[2 * u + 1]);
    }
}

__device__ __forceinline__ void kq_finish(float da, float dma, float db, float dmb, const float (&D1)[4],
                                          const float (&D2)[4], float (&acc)[4]) {
    acc[0] = fmaf(da, D1[0], acc[0]);
    acc[1] = fmaf(da, D1[1], acc[1]);
    acc[2] = fmaf(db, D1[2], acc[2]);
    acc[3] = fmaf(db, D1[3], acc[3]);
    acc[0] = fmaf(-dma, D2[0], acc[0]);
    acc[1] = fmaf(-dma, D2[1], acc[1]);
    acc[2] = fmaf(-dmb, D2[2], acc[2]);
    acc[3] = fmaf(-dmb, D2[3], acc[3]);
}

// Q4_K (144 B: d | dmin | 12 scale bytes | 128 code bytes), lead 0, rows 144
// bytes apart. Lane c's sub-blocks c and c + 4: code bytes 16 + 32 (c / 2)
// (+ 64), nibble c % 2; a high nibble is masked in place (1024 + 16 q) and
// f = 1/16 takes the 16 out.
__device__ __forceinline__ void q4k_row_subs(uint32_t r, uint32_t selc, uint32_t f, uint32_t nf, KqSub (&o)[2],
                                             float& d, float& dmin) {
    uint32_t w[4];
    mvh_lds_v4(r, w);  // d | dmin, scale bytes 0..3, 4..7, 8..11
    // sub-block c: scale = b[c] & 63, min = b[c + 4] & 63; sub-block c + 4:
    // the low / high nibble of b[c + 8] and the top two bits of b[c] / b[c + 4]
    const uint32_t sc0 = w[1] & 0x3F3F3F3Fu, m0 = w[2] & 0x3F3F3F3Fu;
    const uint32_t sc1 = (w[3] & 0x0F0F0F0Fu) | ((w[1] & 0xC0C0C0C0u) >> 2);
    const uint32_t m1 = ((w[3] >> 4) & 0x0F0F0F0Fu) | ((w[2] & 0xC0C0C0C0u) >> 2);
    o[0] = kq_sub(sc0, m0, selc, f, nf);
    o[1] = kq_sub(sc1, m1, selc, f, nf);
    d = half_bits_to_float(w[0] & 0xFFFFu);
    dmin = half_bits_to_float(w[0] >> 16);
}

__device__ __forceinline__ void q4k_stage(uint32_t slot, int g, int c, uint32_t selc, const uint16_t* xr,
                                          float (&acc)[4]) {
    const bool high = (c & 1) != 0;
    const uint32_t nm = high ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    const uint32_t f = high ? kH2Sixteenth : kH2One, nf = high ? kH2M64 : kH2M1024;
    const uint32_t pa = slot + kMvhRow32 * static_cast<uint32_t>(g), pb = pa + 8u * kMvhRow32;
    KqSub sa[2], sb[2];
    float da, dma, db, dmb;
    q4k_row_subs(pa, selc, f, nf, sa, da, dma);
    q4k_row_subs(pb, selc, f, nf, sb, db, dmb);
    float D1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, D2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t co = 16u + 32u * static_cast<uint32_t>(c >> 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            uint32_t wa[4], wb[4];
            mvh_lds_v4(pa + co + 64u * h + 16u * v, wa);
            mvh_lds_v4(pb + co + 64u * h + 16u * v, wb);
            const int x0 = 32 * (c + 4 * h) + 16 * v;
            kq_mma4(wa, wb, nm, sa[h], sb[h], mvh_x8(xr, x0), mvh_x8(xr, x0 + 8), D1, D2);
        }
    }
    kq_finish(da, dma, db, dmb, D1, D2, acc);
}

// Q2_K (84 B: 16 scale bytes | 64 code bytes | d | dmin) at lead L (0, 4, 8
// or 12), rows 96 bytes apart. Lane c's sub-blocks c + 4t: scale byte c of
// scale word t, codes 16 bytes at 16 + 32 (t / 2) + 16 (c % 2), the 2-bit
// field s = c / 2 + 2 (t % 2) of each byte, masked in place (1024 + 4^s q)
// with f = 4^-s. Kept out of line (inlined, it made the kernel spill) and
// returns the stage's sums d D1 - dmin D2 of the lane's four outputs.
__device__ __noinline__ float4 q2k_stage(uint32_t slot, int g, int c, uint32_t L, uint32_t selc,
                                         const uint16_t* xr) {
    const uint32_t s0 = static_cast<uint32_t>(c >> 1);  // field of the even t (0 or 1); odd t: s0 + 2
    const uint32_t pa = slot + kMvhRowQ2K * static_cast<uint32_t>(g) + L, pb = pa + 8u * kMvhRowQ2K;
    float D1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, D2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t co = 16u + 16u * static_cast<uint32_t>(c & 1);
#pragma unroll
    for (int run = 0; run < 2; ++run) {
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            wa[u] = lds_u32(pa + co + 32u * run + 4u * u);
            wb[u] = lds_u32(pb + co + 32u * run + 4u * u);
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const int t = 2 * run + tt;
            const uint32_t f = tt ? (s0 ? kH2Sixtyfourth : kH2Sixteenth) : (s0 ? kH2Quarter : kH2One);
            const uint32_t nf = tt ? (s0 ? kH2M16 : kH2M64) : (s0 ? kH2M256 : kH2M1024);
            const uint32_t ka = lds_u32(pa + 4u * t), kb = lds_u32(pb + 4u * t);
            const KqSub sa = kq_sub(ka & 0x0F0F0F0Fu, (ka >> 4) & 0x0F0F0F0Fu, selc, f, nf);
            const KqSub sb = kq_sub(kb & 0x0F0F0F0Fu, (kb >> 4) & 0x0F0F0F0Fu, selc, f, nf);
            const int x0 = 16 * (c + 4 * t);
            kq_mma4(wa, wb, 0x03030303u << (2u * s0 + 4u * tt), sa, sb, mvh_x8(xr, x0), mvh_x8(xr, x0 + 8), D1,
                    D2);
        }
    }
    const uint32_t dda = lds_u32(pa + 80u), ddb = lds_u32(pb + 80u);
    float r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    kq_finish(half_bits_to_float(dda & 0xFFFFu), half_bits_to_float(dda >> 16), half_bits_to_float(ddb & 0xFFFFu),
              half_bits_to_float(ddb >> 16), D1, D2, r);
    return make_float4(r[0], r[1], r[2], r[3]);
}

// ------------------------------------------------------------ the kernel

__host__ __device__ constexpr int mvh_stage_k(int fmt) { return fmt == FMT_Q8_0 ? 128 : 256; }
__host__ __device__ constexpr int mvh_stage_bytes(int fmt) {
    return fmt == FMT_Q6_K ? 210 : (fmt == FMT_Q4_0 || fmt == FMT_Q4_K) ? 144 : (fmt == FMT_Q2_K ? 84 : 136);
}

// The walk of a warp's (or team's) stages. Teams (KS > 1) take items t,
// t + T, ... (T teams) and member m the stages m, m + KS, ... of each. Single
// warps (KS == 1) take item w (their number in the grid) first, then the next
// unclaimed item of a counter in global memory (reset by the prep kernel),
// so that items of very different lengths (a mixed-format launch) spread
// evenly; each item is still summed by one warp in stage order.
struct MvhCursor {
    int it, p, m;
    bool fetch;  // the item ended; the next one is claimed before the next copy
};

__device__ __forceinline__ void mvh_set_matrix(const MvhGroup& g, MvhCursor& c) {
    while (c.m + 1 < g.nmat && c.it >= g.m[c.m + 1].item0) ++c.m;
}

__device__ __forceinline__ void mvh_advance(const MvhGroup& g, int ks, int member, int nteams, MvhCursor& c) {
    c.p += ks;
    if (c.p < g.m[c.m].stages) return;
    if (ks == 1) {
        c.fetch = true;
        return;
    }
    c.p = member;
    c.it += nteams;
    mvh_set_matrix(g, c);
}

// byte offset of stage p of row j (of every group) in a view row of W
__device__ __forceinline__ int64_t mvh_stage_off(const MvhMat& a, int j, int p) {
    return static_cast<int64_t>(j) * a.rowbytes + static_cast<int64_t>(p) * a.stage_bytes;
}

// Issues the TMA copies of the stage at cursor c into `slot` (completing on
// bar): lane k issues box k, from the 16-byte boundary at or below the
// stage's first byte.
__device__ __forceinline__ void mvh_issue(const MvhGroup& g, const MvhCursor& c, uint32_t slot, uint32_t bar,
                                          int lane) {
    const MvhMat& a = g.m[c.m];
    const int li = c.it - a.item0;
    const int j = li & 7, G0 = (li >> 3) * kMvhRows;
    const int nb = a.boxes;
    const uint32_t bw = static_cast<uint32_t>(a.box_w);
    const int64_t off = mvh_stage_off(a, j, c.p) & ~static_cast<int64_t>(15);
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb) * bw * kMvhRows);
    __syncwarp();
    if (lane < nb)
        tma_load_2d(slot + static_cast<uint32_t>(lane) * bw * kMvhRows, &g.map[c.m],
                    static_cast<int>(off / 2) + static_cast<int>(bw / 2) * lane, G0, bar);
}

// The lane's activation row (xb: its batch row) at the first K of stage p.
__device__ __forceinline__ const uint16_t* mvh_xrow(const MvhMat& a, int xb, int p) {
    return a.xh + static_cast<int64_t>(xb) * a.K + static_cast<int64_t>(p) * a.stage_k;
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

// KQ: the launch has Q4_K / Q2_K matrices. Their stages are built only into
// that instantiation, so the code of the other formats' launches is the same
// as if they did not exist.
template <bool KQ>
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
    int* fifo = reinterpret_cast<int*>(smem + kMvhFifoOff) + 4 * warp;
    const int nteams = static_cast<int>(gridDim.x) * (kMvhWarps / ks);
    const int gt = team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    // byte selector: byte c of a word into the low bytes of two fp16 (1024 + byte)
    const uint32_t selc = 0x4040u | (static_cast<uint32_t>(c) << 8) | static_cast<uint32_t>(c);
    Q6Off po;
    po.o[0] = q6k_poff(c);
    po.o[1] = q6k_poff(c + 1);
    po.o[2] = q6k_poff(4 + c);
    po.o[3] = q6k_poff(5 + c);
    po.o[4] = q6k_poff(8 + c);
    po.o[5] = q6k_poff(9 + c);
    const int xrow_b = gr % g.B;  // a lane past the batch reads a valid row (never stored)

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (gt >= g.items) return;  // the whole team: every member has the same items
    if (lane < kMvhNS) mbar_init(bars + 8 * lane, 1);
    fence_mbar_init();
    __syncwarp();

    // The weights do not depend on the previous kernel: the first copies (of
    // the first item only: later items may come from the counter, which the
    // previous kernel resets) go out before waiting for it.
    MvhCursor ic{gt, member, 0, false};
    mvh_set_matrix(g, ic);
    const int m0 = ic.m;
    uint32_t issued = 0, used = 0;
    int fifo_head = 0, fifo_tail = 0;
    for (int j = 0; j < kMvhNS - 1 && !ic.fetch; ++j) {
        mvh_issue(g, ic, ring + (issued % kMvhNS) * kMvhSlot, bars + 8 * (issued % kMvhNS), lane);
        ++issued;
        mvh_advance(g, ks, member, nteams, ic);
    }
    grid_dependency_wait();  // x and the counter come from the prep kernel
    const int first_claim = static_cast<int>(gridDim.x) * kMvhWarps;

    bool ok = true;
    int m = m0;
    int it = gt;
    while (it < g.items) {
        while (m + 1 < g.nmat && it >= g.m[m + 1].item0) ++m;  // items only increase
        const MvhMat& a = g.m[m];
        const int li = it - a.item0;
        const int j = li & 7, G0 = (li >> 3) * kMvhRows;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int p = member; p < a.stages; p += ks) {
            // the next item of a single warp's walk, claimed once the
            // copies have reached the end of the current one
            if (ic.fetch) {
                int nx = 0;
                if (lane == 0) nx = first_claim + atomicAdd(g.ctr, 1);
                nx = __shfl_sync(0xffffffffu, nx, 0);
                ic.it = nx;
                ic.p = 0;
                ic.fetch = false;
                mvh_set_matrix(g, ic);
                if (lane == 0) fifo[fifo_tail & 3] = nx;
                ++fifo_tail;
            }
            // the copies NS - 1 stages ahead, into the slot consumed last
            if (ic.it < g.items) {
                fence_proxy_async_smem();
                __syncwarp();
                mvh_issue(g, ic, ring + (issued % kMvhNS) * kMvhSlot, bars + 8 * (issued % kMvhNS), lane);
                ++issued;
                mvh_advance(g, ks, member, nteams, ic);
            }
            const uint16_t* xr = mvh_xrow(a, xrow_b, p);
            const uint32_t slot = ring + (used % kMvhNS) * kMvhSlot;
            if (ok) ok = mvh_wait(bars + 8 * (used % kMvhNS), (used / kMvhNS) & 1u, g.st.err);
            ++used;
            const uint32_t L = static_cast<uint32_t>(mvh_stage_off(a, j, p) & 15);
            if (a.fmt == FMT_Q6_K) q6k_stage(slot, gr, c, po, L, selc, xr, acc);
            else if (a.fmt == FMT_Q4_0) q4_0_stage(slot, gr, c, xr, acc);
            else if (!KQ || a.fmt == FMT_Q8_0) q8_0_stage(slot, gr, c, L, xr, acc);
            else if (a.fmt == FMT_Q4_K) q4k_stage(slot, gr, c, selc, xr, acc);
            else {
                const float4 r = q2k_stage(slot, gr, c, L, selc, xr);
                acc[0] += r.x;
                acc[1] += r.y;
                acc[2] += r.z;
                acc[3] += r.w;
            }
            __syncwarp();
        }
        // the team's sums of the item, added by member 0 in member order
        if (ks > 1) {
#pragma unroll
            for (int q = 0; q < 4; ++q) part[(warp * 4 + q) * 32 + lane] = acc[q];
            mvh_team_sync(team, ks);
            if (member == 0) {
                for (int t2 = 1; t2 < ks; ++t2)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[q] += part[((warp + t2) * 4 + q) * 32 + lane];
            }
            mvh_team_sync(team, ks);  // the partial sums are read before they are overwritten
        }
        if (member == 0) {
            // lane (g, c): item rows g and g + 8, batch rows 2c, 2c + 1
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
                const int b = 2 * c + b2;
                if (b >= g.B) continue;
                const float sc = a.xinv[b];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t n = static_cast<int64_t>(j) + 8 * (G0 + gr + 8 * h);
                    if (n < a.N) a.y[static_cast<int64_t>(b) * a.N + n] = acc[2 * h + b2] * sc;
                }
            }
        }
        if (ks > 1) {
            it += nteams;
        } else {
            __syncwarp();  // the cursor's lane 0 wrote the next item before this
            it = fifo[fifo_head & 3];
            ++fifo_head;
        }
    }
    // a slot whose wait gave up may still be receiving: wait for it (bounded)
    // before the CTA's shared memory is released
    if (!ok)
        for (uint32_t u = used > kMvhNS ? used - kMvhNS : 0; u < issued; ++u)
            (void)mvh_wait(bars + 8 * (u % kMvhNS), (u / kMvhNS) & 1u, g.st.err);
}

}  // namespace qmm
