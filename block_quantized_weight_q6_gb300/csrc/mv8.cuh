// mv8.cuh -- fused dequantize + matvec for 2..8 bf16 activation rows (float
// mode) on the warp-level tensor-core MMA (mma.sync m16n8k16, bf16 operands,
// fp32 accumulators):
//
//   y[b][n] = sum_k w[n][k] * x[b][k],   b < B <= 8
//
// Why a warp-level MMA: with 8 activation rows every weight takes 8 FMAs on
// the CUDA cores, more than the FP32 pipe can give at HBM speed, while the
// tensor-memory matvec spends most of its issue slots on handing stages
// between warps. Here each warp decodes its weights straight into MMA
// fragments in registers and multiplies them itself: no tensor memory, no
// barriers between warps.
//
// One MMA takes a 16-row x 16-K tile of exact integer codes as A (bf16: q - 8,
// q, q - 32), the 16 K x 8 activation rows as B and adds into a 16 x 8 fp32
// tile. The 16 K of an MMA are one q6_K scale group, or one half of a Q4_0 /
// Q8_0 block, so the tile's sum is scaled once (by d * sc or d) into the
// lane's accumulators. Lane (g = lane / 4, c = lane % 4) holds rows g and
// g + 8 of a tile; the four K slots it feeds (2c, 2c + 1, 2c + 8, 2c + 9 in
// the MMA's numbering) are given the weights 4c .. 4c + 3 of the 16 and the
// activations of the same four K, so a lane reads four consecutive code
// bytes and one 8-byte run of activations per row and K step.
//
// Work item: 32 rows (two tiles) of one matrix, all of K, in stages of 256
// K; each warp streams its own items through a private ring of stages in
// shared memory (cp.async, as mv1), and loads each stage's activation
// fragments (16 K steps x 8 bytes per lane) one stage ahead.
#pragma once

#include "mv1.cuh"

namespace qmm {

constexpr int kMv8StageK = 256;
constexpr int kMv8RB = kMv8RowBlock;  // rows per item
constexpr int kMv8Warps = 8;

// Per format: bytes of a row's stage (one super-block, or 8 blocks), row
// stride in a stage slot, ring stages per warp.
template <int FMT>
struct Mv8F;
template <>
struct Mv8F<FMT_Q4_0> {
    static constexpr int PB = 8 * 18, RS = PB, NS = 4;
};
template <>
struct Mv8F<FMT_Q8_0> {
    static constexpr int PB = 8 * 34, RS = PB, NS = 3;
};
template <>
struct Mv8F<FMT_Q6_K> {
    // the 16-byte pieces that cover a 210-byte super-block: at most 224 bytes
    static constexpr int PB = 210, RS = 240, NS = 3;
};

// the rings, then the members' sums of an item (8 floats per lane and warp)
template <int FMT>
constexpr uint32_t mv8_smem_bytes() {
    return static_cast<uint32_t>(kMv8Warps * Mv8F<FMT>::NS * kMv8RB * Mv8F<FMT>::RS + kMv8Warps * 8 * 32 * 4);
}
static_assert(mv8_smem_bytes<FMT_Q4_0>() <= 227 * 1024 && mv8_smem_bytes<FMT_Q8_0>() <= 227 * 1024 &&
                  mv8_smem_bytes<FMT_Q6_K>() <= 227 * 1024,
              "shared memory");

// D = A B + C, m16n8k16, bf16 A (row) and B (col), fp32 C and D
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// code bytes (below 128) 0, 1 / 2, 3 of w -> bf16 pairs (128 + code)
__device__ __forceinline__ uint32_t mv8_pair01(uint32_t w) { return __byte_perm(w, 0x43434343u, 0x4140); }
__device__ __forceinline__ uint32_t mv8_pair23(uint32_t w) { return __byte_perm(w, 0x43434343u, 0x4342); }

// v + c on bf16 pairs, one rounding (exact here: small integers)
__device__ __forceinline__ uint32_t mv8_bf_add(uint32_t v, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(0x3F803F80u), "r"(c));
    return d;
}

// A fragment of one K step from the two rows' four code bytes (codes below
// 128; `off` the bf16 pair that subtracts the format's offset)
__device__ __forceinline__ void mv8_afrag(uint32_t ca, uint32_t cb, uint32_t off, uint32_t (&a)[4]) {
    a[0] = mv8_bf_add(mv8_pair01(ca), off);  // row g,     K slots 2c, 2c + 1
    a[1] = mv8_bf_add(mv8_pair01(cb), off);  // row g + 8
    a[2] = mv8_bf_add(mv8_pair23(ca), off);  // row g,     K slots 2c + 8, 2c + 9
    a[3] = mv8_bf_add(mv8_pair23(cb), off);  // row g + 8
}

// Q8_0: signed code bytes -> A fragment, through exact fp32 values whose
// upper halves are the bf16 codes
__device__ __forceinline__ void mv8_q8_pairs(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = w ^ 0x80808080u;  // q + 128, as unsigned bytes
    const float2 neg = make_float2(-(8388608.0f + 128.0f), -(8388608.0f + 128.0f));
    const float2 f01 = fadd2(make_float2(byte_as_magic_float<0>(u), byte_as_magic_float<1>(u)), neg);
    const float2 f23 = fadd2(make_float2(byte_as_magic_float<2>(u), byte_as_magic_float<3>(u)), neg);
    p01 = __byte_perm(__float_as_uint(f01.x), __float_as_uint(f01.y), 0x7632);
    p23 = __byte_perm(__float_as_uint(f23.x), __float_as_uint(f23.y), 0x7632);
}

// four bytes at a 2-byte-aligned shared address
__device__ __forceinline__ uint32_t mv8_lds_w(uint32_t a) {
    const uint32_t lo = lds_u32(a & ~3u), hi = lds_u32((a & ~3u) + 4);
    return __funnelshift_r(lo, hi, 8u * (a & 3u));
}

// ------------------------------------------------------------ one stage
// Adds one tile's products of a stage into acc (D layout: acc[0], acc[1] row
// g, activation rows 2c, 2c + 1; acc[2], acc[3] row g + 8). ra / rb: shared
// address of the stage's bytes of rows g and g + 8 of the tile; xb[s]: the
// lane's activations of K step s (k = 16 s + 4c .. + 3 of the stage).

constexpr uint32_t kMv8Neg136 = 0xC308C308u;  // bf16 pair (-136, -136): (128 + q) - 136 = q - 8
constexpr uint32_t kMv8Neg160 = 0xC320C320u;  // bf16 pair (-160, -160): (128 + q) - 160 = q - 32

// Q4_0: 8 blocks (d fp16 | qs[16]); K step 2b = the low nibbles of block b's
// qs (weights 0..15), step 2b + 1 the high nibbles (16..31); the lane's code
// bytes are qs[4c .. 4c + 3], at 18 b + 2 + 4c (4-byte aligned for odd b).
__device__ __forceinline__ void mv8_stage_q4_0(uint32_t ra, uint32_t rb, int c, const uint2 (&xb)[16],
                                               float (&acc)[4]) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const uint32_t o = 18u * b + 4u * c;
        uint32_t wa, wb;
        if (b & 1) {
            wa = lds_u32(ra + o + 2);
            wb = lds_u32(rb + o + 2);
        } else {
            wa = __byte_perm(lds_u32(ra + o), lds_u32(ra + o + 4), 0x5432);
            wb = __byte_perm(lds_u32(rb + o), lds_u32(rb + o + 4), 0x5432);
        }
        const float da = half_bits_to_float(lds_u16(ra + 18u * b));
        const float db = half_bits_to_float(lds_u16(rb + 18u * b));
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t A[4];
        mv8_afrag(wa & 0x0F0F0F0Fu, wb & 0x0F0F0F0Fu, kMv8Neg136, A);
        mma_bf16_16816(D, A, xb[2 * b].x, xb[2 * b].y);
        mv8_afrag((wa >> 4) & 0x0F0F0F0Fu, (wb >> 4) & 0x0F0F0F0Fu, kMv8Neg136, A);
        mma_bf16_16816(D, A, xb[2 * b + 1].x, xb[2 * b + 1].y);
        acc[0] = fmaf(da, D[0], acc[0]);
        acc[1] = fmaf(da, D[1], acc[1]);
        acc[2] = fmaf(db, D[2], acc[2]);
        acc[3] = fmaf(db, D[3], acc[3]);
    }
}

// Q8_0: 8 blocks (d fp16 | qs[32] int8); step 2b = qs[0..15] of block b,
// 2b + 1 = qs[16..31]; the lane's bytes at 34 b + 2 + 4c (+ 16).
__device__ __forceinline__ void mv8_stage_q8_0(uint32_t ra, uint32_t rb, int c, const uint2 (&xb)[16],
                                               float (&acc)[4]) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const float da = half_bits_to_float(lds_u16(ra + 34u * b));
        const float db = half_bits_to_float(lds_u16(rb + 34u * b));
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t o = 34u * b + 2u + 16u * h + 4u * c;
            uint32_t wa, wb;
            if (b & 1) {
                wa = lds_u32(ra + o);
                wb = lds_u32(rb + o);
            } else {
                wa = __byte_perm(lds_u32(ra + o - 2), lds_u32(ra + o + 2), 0x5432);
                wb = __byte_perm(lds_u32(rb + o - 2), lds_u32(rb + o + 2), 0x5432);
            }
            uint32_t A[4];
            mv8_q8_pairs(wa, A[0], A[2]);
            mv8_q8_pairs(wb, A[1], A[3]);
            mma_bf16_16816(D, A, xb[2 * b + h].x, xb[2 * b + h].y);
        }
        acc[0] = fmaf(da, D[0], acc[0]);
        acc[1] = fmaf(da, D[1], acc[1]);
        acc[2] = fmaf(db, D[2], acc[2]);
        acc[3] = fmaf(db, D[3], acc[3]);
    }
}

// q6_K: one super-block (ql[128] | qh[64] | scales[16] | d) at a 2-byte-
// aligned address; K step s = scale group s: weights 16 s + j take the ql
// nibble s >> 3 of ql[16 (s & 7) + j] and the 2-bit field s >> 2 of
// qh[16 (s & 3) + j]; the lane's j are 4c .. 4c + 3.
__device__ __forceinline__ void mv8_stage_q6k(uint32_t ra, uint32_t rb, int c, const uint2 (&xb)[16],
                                              float (&acc)[4]) {
    uint32_t qla[8], qlb[8], qha[4], qhb[4], sca[4], scb[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        qla[j] = mv8_lds_w(ra + 16u * j + 4u * c);
        qlb[j] = mv8_lds_w(rb + 16u * j + 4u * c);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        qha[j] = mv8_lds_w(ra + 128u + 16u * j + 4u * c);
        qhb[j] = mv8_lds_w(rb + 128u + 16u * j + 4u * c);
        sca[j] = mv8_lds_w(ra + 192u + 4u * j);
        scb[j] = mv8_lds_w(rb + 192u + 4u * j);
    }
    const float da = half_bits_to_float(lds_u16(ra + 208));
    const float db = half_bits_to_float(lds_u16(rb + 208));
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        const int nsh = 4 * (s >> 3), hsh = 2 * (s >> 2);
        const uint32_t ca = ((qla[s & 7] >> nsh) & 0x0F0F0F0Fu) | (((qha[s & 3] >> hsh) & 0x03030303u) << 4);
        const uint32_t cb = ((qlb[s & 7] >> nsh) & 0x0F0F0F0Fu) | (((qhb[s & 3] >> hsh) & 0x03030303u) << 4);
        uint32_t A[4];
        mv8_afrag(ca, cb, kMv8Neg160, A);
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_bf16_16816(D, A, xb[s].x, xb[s].y);
        const float sa = da * static_cast<float>(static_cast<int8_t>(sca[s >> 2] >> (8 * (s & 3))));
        const float sb = db * static_cast<float>(static_cast<int8_t>(scb[s >> 2] >> (8 * (s & 3))));
        acc[0] = fmaf(sa, D[0], acc[0]);
        acc[1] = fmaf(sa, D[1], acc[1]);
        acc[2] = fmaf(sb, D[2], acc[2]);
        acc[3] = fmaf(sb, D[3], acc[3]);
    }
}

template <int FMT>
__device__ __forceinline__ void mv8_stage(uint32_t ra, uint32_t rb, int c, const uint2 (&xb)[16], float (&acc)[4]) {
    if constexpr (FMT == FMT_Q4_0) mv8_stage_q4_0(ra, rb, c, xb, acc);
    else if constexpr (FMT == FMT_Q8_0) mv8_stage_q8_0(ra, rb, c, xb, acc);
    else mv8_stage_q6k(ra, rb, c, xb, acc);
}

// ------------------------------------------------------------ the kernel
// The warps of a CTA form teams of KS (1, 2, 4 or 8; the host picks it so
// that short matrices still occupy every SM). Team t of the grid takes items
// t, t + T, ... (T teams); member j of the team takes the item's stages j,
// j + KS, ... (256 K each). At the end of an item the members' sums meet in
// shared memory and member 0 adds them in member order (the result does not
// depend on timing) and stores y. Each warp's copies run NS - 1 stages ahead
// through a cursor over its own walk; the activation fragments of its next
// stage are loaded while the current one is decoded.

struct Mv8Cursor {
    int it, p, m;  // item, stage of the item (piece of K), matrix
};

__device__ __forceinline__ void mv8_advance(const Mv1Group& g, int ks, int member, int nteams, Mv8Cursor& c) {
    c.p += ks;
    if (c.p < g.m[c.m].pieces) return;
    c.p = member;
    c.it += nteams;
    while (c.m + 1 < g.nmat && c.it >= g.m[c.m + 1].item0) ++c.m;
}

// Issues the copies of the stage at cursor c (rows past N are not copied).
template <int FMT>
__device__ __forceinline__ void mv8_issue(const Mv1Group& g, const Mv8Cursor& c, uint32_t slot, int lane) {
    using F = Mv8F<FMT>;
    const Mv1Mat& a = g.m[c.m];
    const int64_t row0 = static_cast<int64_t>(c.it - a.item0) * kMv8RB;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kMv8RB), a.N - row0));
    const uint8_t* base = a.W + row0 * a.rowbytes + static_cast<int64_t>(c.p) * F::PB;
    if constexpr (FMT != FMT_Q6_K) {
        // Q4_0 / Q8_0 rows (K % 256 == 0, W 16-byte aligned) are whole
        // 16-byte pieces: the stage's rows one after another
        constexpr int CPR = F::PB / 16;
#pragma unroll
        for (int i = 0; i < (kMv8RB * CPR + 31) / 32; ++i) {
            const int q = lane + 32 * i;
            const int r = q / CPR, cc = q % CPR;
            if (q < kMv8RB * CPR && r < rows)
                cp_async16(slot + static_cast<uint32_t>(r * F::RS + 16 * cc), base + r * a.rowbytes + 16 * cc);
        }
        return;
    }
    // q6_K: the 14 16-byte pieces from the boundary below each row's
    // super-block (rows of whole 16-byte pieces share one start offset);
    // only the matrix's last super-block can end inside its last piece, and
    // is read up to the matrix's end
    constexpr int NP = 14;
    const bool tail = rows == static_cast<int>(a.N - row0) && c.p + 1 == a.pieces;
    const uint8_t* end = a.W + a.N * a.rowbytes;
    if (a.aligned) {
        const uint8_t* start = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(base) & ~uintptr_t{15});
#pragma unroll
        for (int i = 0; i < (kMv8RB * NP + 31) / 32; ++i) {
            const int q = lane + 32 * i;
            const int r = q / NP, cc = q % NP;
            if (r >= rows) continue;
            const uint8_t* s16 = start + r * a.rowbytes + 16 * cc;
            const uint32_t dst = slot + static_cast<uint32_t>(r * F::RS + 16 * cc);
            if (!tail || s16 + 16 <= end) cp_async16(dst, s16);
            else if (s16 < end) cp_async16_part(dst, s16, static_cast<uint32_t>(end - s16));
        }
    } else {
#pragma unroll
        for (int i = 0; i < (kMv8RB * NP + 31) / 32; ++i) {
            const int q = lane + 32 * i;
            const int r = q / NP, cc = q % NP;
            if (r >= rows) continue;
            const uint8_t* start = reinterpret_cast<const uint8_t*>(
                reinterpret_cast<uintptr_t>(base + r * a.rowbytes) & ~uintptr_t{15});
            const uint8_t* s16 = start + 16 * cc;
            const uint32_t dst = slot + static_cast<uint32_t>(r * F::RS + 16 * cc);
            if (!tail || s16 + 16 <= end) cp_async16(dst, s16);
            else if (s16 < end) cp_async16_part(dst, s16, static_cast<uint32_t>(end - s16));
        }
    }
}

// The lane's activation fragments of stage p of matrix a: activation row g
// (zero past B), k = 256 p + 16 s + 4c .. + 3 for s < 16.
__device__ __forceinline__ void mv8_x_fetch(const Mv1Group& g, const Mv1Mat& a, int p, int lane, uint2 (&xb)[16]) {
    const int gr = lane >> 2, c = lane & 3;
    if (gr < g.B) {
        const uint16_t* x = static_cast<const uint16_t*>(a.x) + static_cast<int64_t>(gr) * a.K +
                            static_cast<int64_t>(p) * kMv8StageK + 4 * c;
#pragma unroll
        for (int s = 0; s < 16; ++s) xb[s] = __ldg(reinterpret_cast<const uint2*>(x + 16 * s));
    } else {
#pragma unroll
        for (int s = 0; s < 16; ++s) xb[s] = make_uint2(0u, 0u);
    }
}

// barrier of the team's warps (named barrier 1 + team)
__device__ __forceinline__ void mv8_team_sync(int team, int ks) {
    if (ks > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * ks) : "memory");
}

template <int FMT>
__global__ void __launch_bounds__(kMv8Warps * 32, 1) mv8_kernel(const __grid_constant__ Mv1Group g) {
    using F = Mv8F<FMT>;
    constexpr int NS = F::NS;
    constexpr uint32_t SLOT = kMv8RB * F::RS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, c = lane & 3;
    const int ks = g.ks;
    const int team = warp / ks, member = warp % ks;
    const uint32_t ring = smem_u32(smem) + static_cast<uint32_t>(warp) * NS * SLOT;
    // the members' sums of an item: [warp][8][lane] fp32, after the rings
    float* part = reinterpret_cast<float*>(smem + kMv8Warps * NS * SLOT);
    // teams numbered across CTAs first, so that a second round of items
    // spreads over all SMs
    const int nteams = static_cast<int>(gridDim.x) * (kMv8Warps / ks);
    const int gt = team * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (gt >= g.items) return;  // the whole team: every member has the same items
    // the weights do not depend on the previous kernel: the first copies go
    // out before waiting for it
    Mv8Cursor ic{gt, member, 0};
    while (ic.m + 1 < g.nmat && ic.it >= g.m[ic.m + 1].item0) ++ic.m;
    const int m0 = ic.m;
    int si = 0;
#pragma unroll
    for (int j = 0; j < NS - 1; ++j) {
        if (ic.it < g.items) {
            mv8_issue<FMT>(g, ic, ring + si * SLOT, lane);
            mv8_advance(g, ks, member, nteams, ic);
        }
        cp_async_commit();
        si = si + 1 == NS ? 0 : si + 1;
    }
    grid_dependency_wait();  // x comes from the previous kernel

    uint2 xb[16], xn[16];
    mv8_x_fetch(g, g.m[m0], member, lane, xn);
    int sc = 0;
    int m = m0;
    for (int it = gt; it < g.items; it += nteams) {
        while (m + 1 < g.nmat && it >= g.m[m + 1].item0) ++m;
        const Mv1Mat& a = g.m[m];
        const int64_t row0 = static_cast<int64_t>(it - a.item0) * kMv8RB;
        float acc[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[t][q] = 0.0f;
        for (int p = member; p < a.pieces; p += ks) {
#pragma unroll
            for (int s = 0; s < 16; ++s) xb[s] = xn[s];
            // the next stage's activations (this item's, or the next item's first)
            if (p + ks < a.pieces) {
                mv8_x_fetch(g, a, p + ks, lane, xn);
            } else if (it + nteams < g.items) {
                int mn = m;
                while (mn + 1 < g.nmat && it + nteams >= g.m[mn + 1].item0) ++mn;
                mv8_x_fetch(g, g.m[mn], member, lane, xn);
            }
            if (ic.it < g.items) {
                mv8_issue<FMT>(g, ic, ring + si * SLOT, lane);
                mv8_advance(g, ks, member, nteams, ic);
            }
            cp_async_commit();
            si = si + 1 == NS ? 0 : si + 1;
            cp_async_wait<NS - 1>();
            __syncwarp();
            const uint32_t slot = ring + sc * SLOT;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int ra = 16 * t + gr, rb = ra + 8;
                uint32_t la = 0, lb = 0;
                if constexpr (FMT == FMT_Q6_K) {
                    // offset of each row's super-block in its first 16-byte piece
                    const uintptr_t w0 = reinterpret_cast<uintptr_t>(a.W) + static_cast<int64_t>(p) * F::PB;
                    la = static_cast<uint32_t>((w0 + (row0 + ra) * a.rowbytes) & 15);
                    lb = static_cast<uint32_t>((w0 + (row0 + rb) * a.rowbytes) & 15);
                }
                mv8_stage<FMT>(slot + ra * F::RS + la, slot + rb * F::RS + lb, c, xb, acc[t]);
            }
            __syncwarp();
            sc = sc + 1 == NS ? 0 : sc + 1;
        }
        // the team's sums of the item, added by member 0 in member order
        if (ks > 1) {
#pragma unroll
            for (int q = 0; q < 8; ++q) part[(warp * 8 + q) * 32 + lane] = acc[q >> 2][q & 3];
            mv8_team_sync(team, ks);
            if (member == 0) {
                for (int j = 1; j < ks; ++j)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q >> 2][q & 3] += part[((warp + j) * 8 + q) * 32 + lane];
            }
            mv8_team_sync(team, ks);  // the partial sums are read before they are overwritten
        }
        if (member == 0) {
            // lane (g, c): rows 16 t + g and 16 t + g + 8, activation rows 2c, 2c + 1
#pragma unroll
            for (int t = 0; t < 2; ++t) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t n = row0 + 16 * t + gr + 8 * h;
                    if (n >= a.N) continue;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int b = 2 * c + j;
                        if (b < g.B) a.y[static_cast<int64_t>(b) * a.N + n] = acc[t][2 * h + j];
                    }
                }
            }
        }
    }
}

}  // namespace qmm
