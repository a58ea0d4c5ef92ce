// mv1.cuh -- fused dequantize + matvec for ONE activation row (batch 1, float
// mode) on the CUDA cores:
//
//   y[n] = sum_k w[n][k] * x[k],   w = d * (q - 8) | d * q | d * sc * (q - 32)
//
// Why not the tensor cores here: at batch 1 every weight meets one
// activation, so the multiply is a single packed FMA per two weights. What
// costs is the unpack and the bookkeeping around it, and a pipeline of
// warps that hand stages to each other spends most of its issue slots on
// that bookkeeping. This kernel has none: every warp streams its own weight
// rows through a private ring of shared-memory stages (cp.async, 16-byte
// pieces, coalesced) and decodes them where they land.
//
// Lanes run along K. K is cut into pieces of 2048; in a piece, lane l owns
// 64 columns, and holds their 64 activations in registers (fp32) for every
// row it visits, so activations are read once per piece, not once per row:
//   Q4_0 / Q8_0  columns 64 l .. 64 l + 63 (blocks 2 l and 2 l + 1)
//   q6_K         super-block l / 4 of the piece, "columns" 16 (l % 4) .. + 15:
//                column c of a super-block is the four weights c, c + 64,
//                c + 128, c + 192, which share ql bytes c and c + 64 and qh
//                byte c, so a lane reads 16 + 16 + 16 bytes, 4 scales and d
//                and decodes 64 weights in four scale groups (16 (l % 4) + 64 j
//                .. + 15, j = 0..3).
// Work item = (matrix, block of RB rows), all pieces in order; a lane sums its
// columns' products of each row over the pieces, and the warp adds the lanes
// of each row at the end of the item (butterfly, fixed order: the result
// does not depend on timing). A stage is RC rows of one piece.
//
// Unpack: code bytes -> floats 2^23 + byte (one byte-permute each), minus
// 2^23 + offset (one packed add per two weights) = the exact integer code;
// one packed FMA per two weights with the activations; per block or scale
// group the fp32 sum is scaled (d, or sc then d).
#pragma once

#include "kernels.h"

namespace qmm {

constexpr int kMv1PieceK = 2048;  // K per piece: 32 lanes x 64 columns

// Per format: block bytes, bytes of one row's piece (full), the row's stride
// in a stage, stage rows, ring stages per warp. Q4_0 / Q8_0 rows (K % 256 ==
// 0) are whole 16-byte pieces; a q6_K row need not be (210-byte blocks), so
// its piece is copied as the 16-byte pieces that cover it and decoded from
// its offset ("lead", even, below 16) in the first one.
template <int FMT>
struct Mv1F;
template <>
struct Mv1F<FMT_Q4_0> {
    static constexpr int BB = 18, PB = 64 * 18, RS = PB, RC = 4, NS = 4;
};
template <>
struct Mv1F<FMT_Q8_0> {
    static constexpr int BB = 34, PB = 64 * 34, RS = PB, RC = 2, NS = 3;
};
template <>
struct Mv1F<FMT_Q6_K> {
    static constexpr int BB = 210, PB = 8 * 210, RS = PB + 32, RC = 2, NS = 4;
};

constexpr int kMv1Warps = 12;
constexpr int kMv1RB = kMv1RowBlock;  // rows per work item

static_assert(kMv1Warps * Mv1F<FMT_Q4_0>::NS * Mv1F<FMT_Q4_0>::RC * Mv1F<FMT_Q4_0>::RS <= 227 * 1024 &&
                  kMv1Warps * Mv1F<FMT_Q8_0>::NS * Mv1F<FMT_Q8_0>::RC * Mv1F<FMT_Q8_0>::RS <= 227 * 1024 &&
                  kMv1Warps * Mv1F<FMT_Q6_K>::NS * Mv1F<FMT_Q6_K>::RC * Mv1F<FMT_Q6_K>::RS <= 227 * 1024,
              "shared memory");

template <int FMT>
constexpr uint32_t mv1_smem_bytes() {
    return static_cast<uint32_t>(kMv1Warps * Mv1F<FMT>::NS * Mv1F<FMT>::RC * Mv1F<FMT>::RS);
}

// 16-byte copy global -> shared, through L2 only; a miss fetches the 256
// bytes around it from HBM (a row's piece is read whole, in order)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// the same, reading only the first `bytes` (< 16) of the source and filling
// the rest with zeros
__device__ __forceinline__ void cp_async16_part(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------ activations
// The 64 activations of lane `lane` in piece p, as the order the decoders
// use: Q4_0 / Q8_0 k = 2048 p + 64 lane + i; q6_K k = 2048 p + 256 (lane / 4)
// + 64 j + 16 (lane % 4) + i (i < 16, j < 4, stored at 16 j + i). Columns at
// or past K read as zero.
template <int FMT>
__device__ __forceinline__ int64_t mv1_xrun(int64_t p, int lane, int run) {
    // first k of run `run` (0..3) of 16 consecutive activations
    if constexpr (FMT == FMT_Q6_K)
        return p * kMv1PieceK + 256 * (lane >> 2) + 64 * run + 16 * (lane & 3);
    else
        return p * kMv1PieceK + 64 * lane + 16 * run;
}

// bf16 activations: raw words (two bf16 each) of the four runs, fetched ahead
template <int FMT>
__device__ __forceinline__ void mv1_x_fetch_bf16(const uint16_t* x, int64_t K, int64_t p, int lane,
                                                 uint4 (&raw)[8]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t k = mv1_xrun<FMT>(p, lane, r);
        if (k < K) {
            const uint4* src = reinterpret_cast<const uint4*>(x + k);
            raw[2 * r] = __ldg(src);
            raw[2 * r + 1] = __ldg(src + 1);
        } else {
            raw[2 * r] = make_uint4(0, 0, 0, 0);
            raw[2 * r + 1] = make_uint4(0, 0, 0, 0);
        }
    }
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ void mv1_x_from_bf16(const uint4 (&raw)[8], float2 (&xf)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        xf[4 * i] = bf16x2_to_float2(raw[i].x);
        xf[4 * i + 1] = bf16x2_to_float2(raw[i].y);
        xf[4 * i + 2] = bf16x2_to_float2(raw[i].z);
        xf[4 * i + 3] = bf16x2_to_float2(raw[i].w);
    }
}

template <int FMT>
__device__ __forceinline__ void mv1_x_load_f32(const float* x, int64_t K, int64_t p, int lane,
                                               float2 (&xf)[32]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t k = mv1_xrun<FMT>(p, lane, r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < K) v = __ldg(reinterpret_cast<const float4*>(x + k) + i);
            xf[8 * r + 2 * i] = make_float2(v.x, v.y);
            xf[8 * r + 2 * i + 1] = make_float2(v.z, v.w);
        }
    }
}

// ------------------------------------------------------------ decoders
// Each returns lane `lane`'s sum over its 64 columns of one row, from the
// row's piece at shared address `row` (the piece's first byte).

// Q4_0 block (d fp16 | qs[16]); qs byte j holds weights j (low nibble) and
// j + 16 (high nibble), w = d * (q - 8). The lane's two blocks start at
// 36 lane (4-byte aligned): block 0's qs at bytes 2..17, block 1's at 20..35.
// (Masking each nibble straight into a magic float's mantissa, four scales
// in four accumulator lanes, costs fewer instructions but ran slower here.)
__device__ __forceinline__ float mv1_dec_q4_0(uint32_t row, int lane, const float2 (&x)[32]) {
    const uint32_t a = row + 36u * static_cast<uint32_t>(lane);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = lds_u32(a + 4 * i);
    uint32_t lo[9], hi[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        lo[i] = w[i] & 0x0F0F0F0Fu;
        hi[i] = (w[i] >> 4) & 0x0F0F0F0Fu;
    }
    const float2 neg = make_float2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
    float r = 0.0f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int p0 = 18 * b;
        const uint32_t dbits = (p0 & 3) == 0 ? (w[p0 >> 2] & 0xFFFFu) : (w[p0 >> 2] >> 16);
        float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const int pa = p0 + 2 + j;  // even: the pair shares a word
            const int wi = pa >> 2, bj = pa & 3;
            const float2 ql = fadd2(make_float2(__uint_as_float(__byte_perm(lo[wi], 0x4B000000u, 0x7540u + bj)),
                                                __uint_as_float(__byte_perm(lo[wi], 0x4B000000u, 0x7541u + bj))),
                                    neg);
            const float2 qh = fadd2(make_float2(__uint_as_float(__byte_perm(hi[wi], 0x4B000000u, 0x7540u + bj)),
                                                __uint_as_float(__byte_perm(hi[wi], 0x4B000000u, 0x7541u + bj))),
                                    neg);
            s0 = ffma2(ql, x[16 * b + j / 2], s0);
            s1 = ffma2(qh, x[16 * b + 8 + j / 2], s1);
        }
        const float2 s = fadd2(s0, s1);
        r = fmaf(half_bits_to_float(dbits), s.x + s.y, r);
    }
    return r;
}

// Q8_0 block (d fp16 | qs[32] int8), w = d * q. The lane's two blocks start
// at 68 lane: block 0's qs at bytes 2..33, block 1's at 36..67.
__device__ __forceinline__ float mv1_dec_q8_0(uint32_t row, int lane, const float2 (&x)[32]) {
    const uint32_t a = row + 68u * static_cast<uint32_t>(lane);
    uint32_t u[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) u[i] = lds_u32(a + 4 * i) ^ 0x80808080u;  // q + 128 as unsigned bytes
    const float2 neg = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    float r = 0.0f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int p0 = 34 * b;
        // d's bytes were flipped with the codes; flip them back
        const uint32_t dw = u[p0 >> 2] ^ 0x80808080u;
        const uint32_t dbits = (p0 & 3) == 0 ? (dw & 0xFFFFu) : (dw >> 16);
        float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const int pa = p0 + 2 + j;
            const int wi = pa >> 2, bj = pa & 3;
            const float2 q = fadd2(make_float2(__uint_as_float(__byte_perm(u[wi], 0x4B000000u, 0x7540u + bj)),
                                               __uint_as_float(__byte_perm(u[wi], 0x4B000000u, 0x7541u + bj))),
                                   neg);
            if ((j & 2) == 0)
                s0 = ffma2(q, x[16 * b + j / 2], s0);
            else
                s1 = ffma2(q, x[16 * b + j / 2], s1);
        }
        const float2 s = fadd2(s0, s1);
        r = fmaf(half_bits_to_float(dbits), s.x + s.y, r);
    }
    return r;
}

// q6_K super-block (ql[128] | qh[64] | scales[16] int8 | d fp16), weight i:
// q = (ql[i & 127] >> 4 (i >> 7)) & 15 | ((qh[i & 63] >> 2 (i >> 6)) & 3) << 4,
// w = d * scales[i >> 4] * (q - 32). The lane's super-block starts at
// 210 (lane / 4) of the piece (2-byte aligned), its columns at 16 (lane % 4).
__device__ __forceinline__ float mv1_dec_q6k(uint32_t row, int lane, const float2 (&x)[32]) {
    const uint32_t sb = row + 210u * static_cast<uint32_t>(lane >> 2);
    const uint32_t cq = static_cast<uint32_t>(lane & 3);
    uint32_t A[4], B[4], H[4];
    lds_words_unaligned<4>(sb + 16 * cq, A);        // ql[c], low nibbles: quarter 0; high: quarter 2
    lds_words_unaligned<4>(sb + 64 + 16 * cq, B);   // ql[c + 64]: quarters 1 and 3
    lds_words_unaligned<4>(sb + 128 + 16 * cq, H);  // qh[c]: 2 bits per quarter
    float sc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sc[j] = static_cast<float>(lds_s8(sb + 192 + cq + 4 * j));
    const float d = half_bits_to_float(lds_u16(sb + 208));
    const float2 neg = make_float2(-8388640.0f, -8388640.0f);  // -(2^23 + 32)
    float r = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint32_t c;
            if (j == 0) c = (A[t] & 0x0F0F0F0Fu) | ((H[t] & 0x03030303u) << 4);
            else if (j == 1) c = (B[t] & 0x0F0F0F0Fu) | ((H[t] & 0x0C0C0C0Cu) << 2);
            else if (j == 2) c = ((A[t] >> 4) & 0x0F0F0F0Fu) | (H[t] & 0x30303030u);
            else c = ((B[t] >> 4) & 0x0F0F0F0Fu) | ((H[t] >> 2) & 0x30303030u);
            const float2 c01 = fadd2(make_float2(byte_as_magic_float<0>(c), byte_as_magic_float<1>(c)), neg);
            const float2 c23 = fadd2(make_float2(byte_as_magic_float<2>(c), byte_as_magic_float<3>(c)), neg);
            s = ffma2(c01, x[8 * j + 2 * t], s);
            s = ffma2(c23, x[8 * j + 2 * t + 1], s);
        }
        r = fmaf(sc[j], s.x + s.y, r);
    }
    return d * r;
}

template <int FMT>
__device__ __forceinline__ float mv1_dec(uint32_t row, int lane, const float2 (&x)[32]) {
    if constexpr (FMT == FMT_Q4_0) return mv1_dec_q4_0(row, lane, x);
    else if constexpr (FMT == FMT_Q8_0) return mv1_dec_q8_0(row, lane, x);
    else return mv1_dec_q6k(row, lane, x);
}

// ------------------------------------------------------------ the kernel
// Warp w of the grid takes items w, w + W, ... (W warps); per item the
// pieces in order, per piece SPP stages of RC rows. The copies run NS - 1
// stages ahead of the decoding, through a cursor over the same walk.

struct Mv1Cursor {
    int it, p, m, u;  // item, piece, matrix, stage of the piece
};

// next stage of the walk; the matrix index only moves forward
template <int SPP>
__device__ __forceinline__ void mv1_advance(const Mv1Group& g, int nw, Mv1Cursor& c) {
    if (++c.u < SPP) return;
    c.u = 0;
    if (++c.p < g.m[c.m].pieces) return;
    c.p = 0;
    c.it += nw;
    while (c.m + 1 < g.nmat && c.it >= g.m[c.m + 1].item0) ++c.m;
}

// Byte offset of row `row`'s piece p from the 16-byte boundary below it.
template <int FMT>
__device__ __forceinline__ uint32_t mv1_lead(const Mv1Mat& a, int64_t row, int p) {
    if constexpr (FMT != FMT_Q6_K) return 0;
    return static_cast<uint32_t>((reinterpret_cast<uintptr_t>(a.W) + row * a.rowbytes +
                                  static_cast<int64_t>(p) * Mv1F<FMT>::PB) & 15);
}

// This lane's 16-byte copies of a full stage (RC rows x a full piece): the
// source offsets from the stage's first byte depend on the row pitch only,
// so they are computed once per matrix (N copies at most; unused entries are
// -1).
template <int FMT>
struct Mv1Copies {
    static constexpr int CPR = Mv1F<FMT>::PB / 16;
    static constexpr int N = (Mv1F<FMT>::RC * CPR + 31) / 32;
    int32_t src[N];
};

template <int FMT>
__device__ __forceinline__ void mv1_copies_init(Mv1Copies<FMT>& cp, int64_t rowbytes, int lane) {
    using C = Mv1Copies<FMT>;
#pragma unroll
    for (int i = 0; i < C::N; ++i) {
        const int q = lane + 32 * i;
        const int r = q / C::CPR, cc = q % C::CPR;
        cp.src[i] = q < Mv1F<FMT>::RC * C::CPR ? static_cast<int32_t>(r * rowbytes + 16 * cc) : -1;
    }
}

// Issues the copies of the stage at cursor c (rows past N are left as they were).
template <int FMT>
__device__ __forceinline__ void mv1_issue(const Mv1Group& g, const Mv1Cursor& c, const Mv1Copies<FMT>& cp,
                                          uint32_t slot, int lane) {
    using F = Mv1F<FMT>;
    using C = Mv1Copies<FMT>;
    const Mv1Mat& a = g.m[c.m];
    const int64_t row0 = static_cast<int64_t>(c.it - a.item0) * kMv1RB + c.u * F::RC;
    const int64_t off = static_cast<int64_t>(c.p) * F::PB;
    const uint8_t* base = a.W + row0 * a.rowbytes + off;
    if (a.aligned && c.p < a.full_pieces && row0 + F::RC <= a.N) {
        // whole 16-byte pieces, as many per row as the format's full piece
#pragma unroll
        for (int i = 0; i < C::N; ++i) {
            const int q = lane + 32 * i;
            const uint32_t dst = static_cast<uint32_t>((q / C::CPR) * F::RS + 16 * (q % C::CPR));
            if (i + 1 < C::N || cp.src[i] >= 0) cp_async16(slot + dst, base + cp.src[i]);
        }
        return;
    }
    // the 16-byte pieces that cover each row's piece; the last piece of the
    // matrix is read only up to its end
    const int rows = static_cast<int>(min(static_cast<int64_t>(F::RC), a.N - row0));
    const uintptr_t end = reinterpret_cast<uintptr_t>(a.W) + static_cast<uintptr_t>(a.N * a.rowbytes);
    const int64_t len = min(static_cast<int64_t>(F::PB), a.rowbytes - off);
    for (int r = 0; r < rows; ++r) {
        const uintptr_t at = reinterpret_cast<uintptr_t>(base + r * a.rowbytes);
        const uintptr_t start = at & ~static_cast<uintptr_t>(15);
        const int n16 = static_cast<int>((at - start + len + 15) / 16);
        for (int cc = lane; cc < n16; cc += 32) {
            const uintptr_t src = start + 16 * cc;
            const uint32_t dst = slot + static_cast<uint32_t>(r * F::RS + 16 * cc);
            if (src + 16 <= end)
                cp_async16(dst, reinterpret_cast<const void*>(src));
            else
                cp_async16_part(dst, reinterpret_cast<const void*>(src), static_cast<uint32_t>(end - src));
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kMv1Warps * 32, 1) mv1_kernel(const __grid_constant__ Mv1Group g) {
    using F = Mv1F<FMT>;
    constexpr int RC = F::RC, NS = F::NS, SPP = kMv1RB / RC;
    constexpr uint32_t SLOT = RC * F::RS;
    static_assert(kMv1RB % RC == 0, "stages per piece");
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem) + static_cast<uint32_t>(warp) * NS * SLOT;
    // warp numbering across CTAs first, so that a second round of items
    // spreads over all SMs
    const int gw = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    const int nw = static_cast<int>(gridDim.x) * kMv1Warps;

    grid_launch_dependents();
    live_bump(g.st, g.live_slot);
    if (gw >= g.items) return;
    // the weights do not depend on the previous kernel: their first copies
    // go out before waiting for it
    Mv1Cursor ic{gw, 0, 0, 0};
    while (ic.m + 1 < g.nmat && ic.it >= g.m[ic.m + 1].item0) ++ic.m;
    const int m0 = ic.m;
    Mv1Copies<FMT> cp;  // this lane's copy offsets for the rows of matrix cp_m
    int cp_m = m0;
    mv1_copies_init<FMT>(cp, g.m[m0].rowbytes, lane);
    auto issue = [&](uint32_t slot) {
        if (ic.m != cp_m) {
            cp_m = ic.m;
            mv1_copies_init<FMT>(cp, g.m[cp_m].rowbytes, lane);
        }
        mv1_issue<FMT>(g, ic, cp, slot, lane);
        mv1_advance<SPP>(g, nw, ic);
    };
    int si = 0;  // ring slot of the next issue
#pragma unroll
    for (int j = 0; j < NS - 1; ++j) {
        if (ic.it < g.items) issue(ring + si * SLOT);
        cp_async_commit();
        si = si + 1 == NS ? 0 : si + 1;
    }
    grid_dependency_wait();  // x comes from the previous kernel

    float2 xf[32];
    uint4 xr[8];
    float acc[kMv1RB];
    int sc = 0;  // ring slot of the next stage to decode
    if (g.x_bf16) mv1_x_fetch_bf16<FMT>(static_cast<const uint16_t*>(g.m[m0].x), g.m[m0].K, 0, lane, xr);
    int m = m0;
    for (int it = gw; it < g.items; it += nw) {
        while (m + 1 < g.nmat && it >= g.m[m + 1].item0) ++m;
        const Mv1Mat& a = g.m[m];
        const int64_t row0 = static_cast<int64_t>(it - a.item0) * kMv1RB;
#pragma unroll
        for (int r = 0; r < kMv1RB; ++r) acc[r] = 0.0f;
        for (int p = 0; p < a.pieces; ++p) {
            // this piece's activations into registers; the next piece's fetched
            if (g.x_bf16) {
                mv1_x_from_bf16(xr, xf);
                const bool last = p + 1 == a.pieces;
                if (!last || it + nw < g.items) {
                    int mn = m;
                    if (last)
                        while (mn + 1 < g.nmat && it + nw >= g.m[mn + 1].item0) ++mn;
                    mv1_x_fetch_bf16<FMT>(static_cast<const uint16_t*>(g.m[mn].x), g.m[mn].K, last ? 0 : p + 1, lane,
                                          xr);
                }
            } else {
                mv1_x_load_f32<FMT>(static_cast<const float*>(a.x), a.K, p, lane, xf);
            }
            // lanes past K in a partial last piece add nothing
            const bool active = static_cast<int64_t>(p) * kMv1PieceK +
                                    (FMT == FMT_Q6_K ? 256 * (lane >> 2) : 64 * lane) < a.K;
#pragma unroll
            for (int u = 0; u < SPP; ++u) {
                if (ic.it < g.items) issue(ring + si * SLOT);
                cp_async_commit();
                si = si + 1 == NS ? 0 : si + 1;
                cp_async_wait<NS - 1>();
                __syncwarp();
                const uint32_t slot = ring + sc * SLOT;
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    const uint32_t lead = mv1_lead<FMT>(a, row0 + u * RC + r, p);
                    const float v = mv1_dec<FMT>(slot + r * F::RS + lead, lane, xf);
                    acc[u * RC + r] += active ? v : 0.0f;
                }
                __syncwarp();
                sc = sc + 1 == NS ? 0 : sc + 1;
            }
        }
        // the item's rows: add the lanes (fixed butterfly), lane r stores row r
#pragma unroll
        for (int r = 0; r < kMv1RB; ++r) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
        }
        float v = acc[0];
#pragma unroll
        for (int r = 1; r < kMv1RB; ++r)
            if (lane == r) v = acc[r];
        if (lane < kMv1RB && row0 + lane < a.N) a.y[row0 + lane] = v;
    }
}

}  // namespace qmm
