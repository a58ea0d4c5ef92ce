// gemv_impl.cuh -- device code of the fused dequantize + matvec kernels,
// included by one translation unit per weight format (gemv_q6k.cu,
// gemv_q4_0.cu, gemv_q8_0.cu) which instantiate it.
//
// Why this shape (quantprobe "LAWS.md", Law 4 amendment L-15 / L-16): decode
// speed is set by the bytes streamed AND by the format's unpack instruction
// cost. So the weights are streamed once, with 1-D bulk TMA copies into a
// per-warp ring of shared-memory slots (many bytes in flight, no per-thread
// load instructions), and the unpack works on whole 32-bit words: four codes
// per bit operation, one byte-permute per code to form its float, and
// packed two-lane fp32 adds and FMAs.
//
// q6_K element expansion ("57 - r54 MINFER_MMQ_Q6K_EXP" section 2.1): every
// 16-element group reads 16 consecutive ql bytes and 16 consecutive qh bytes
// with one shift pair; code = (ql >> qsh & 0xF) | (qh >> qh_shift & 3) << 4.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace qmm {

template <int FMT>
struct Fmt;
template <>
struct Fmt<FMT_Q6_K> {
    static constexpr int BB = 210, BE = 256, CB = 8;
};
template <>
struct Fmt<FMT_Q4_0> {
    static constexpr int BB = 18, BE = 32, CB = 32;
};
template <>
struct Fmt<FMT_Q8_0> {
    static constexpr int BB = 34, BE = 32, CB = 32;
};

// A row segment of one chunk lands at a 16-byte-aligned slot offset with up
// to 15 bytes of lead-in; 32 bytes of slack cover the lead-in and the
// word-granular over-read of the unaligned loads.
template <int FMT>
__host__ __device__ constexpr int seg_stride() {
    return Fmt<FMT>::CB * Fmt<FMT>::BB + 32;
}

static_assert(seg_stride<FMT_Q6_K>() % 16 == 0, "q6_K segment stride");
static_assert(seg_stride<FMT_Q4_0>() % 16 == 0, "Q4_0 segment stride");
static_assert(seg_stride<FMT_Q8_0>() % 16 == 0, "Q8_0 segment stride");

constexpr float kMagic = 8388608.0f;   // 2^23: byte b -> float(2^23 + b)
constexpr int kMagicI = 0x4B400000;    // bits of 1.5 * 2^23: an int32 sum started here
constexpr float kMagicIF = 12582912.0f;  // reads back as a float for |sum| < 2^22

// Two lane mappings:
//  WIDE   (batch rows <= 2): a lane decodes many weights of one block; the
//         activations of the lane's runs are loaded once per chunk and reused
//         for the R rows of the item.
//  NARROW (batch rows >= 4): a lane decodes 8 consecutive weights per pass,
//         so the 32 lanes of a warp read one contiguous run of activations
//         (coalesced) that serves all R rows, and the batch loop is inside.
template <bool Q8, int NB>
struct Wide {
    // int8 activations are 4x smaller than fp32 ones: the hoisted layout
    // stays cheap up to 8 batch rows
    static constexpr bool value = Q8 ? NB <= 8 : NB <= 2;
};

// ------------------------------------------------------------ activations

// 16 activations of batch row b starting at column k0 (multiple of 8) as
// 8 fp32 pairs, from the caller's x (fp32 or bf16)
__device__ __forceinline__ void load_x16(const GemvArgs& a, int b, int64_t k0, float2 (&o)[8]) {
    if (a.x_bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                        b * a.K + k0);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint4 v = __ldg(p + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[4 * i + j] = make_float2(__uint_as_float(w[j] << 16),
                                           __uint_as_float(w[j] & 0xFFFF0000u));
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) +
                                                          b * a.K + k0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = __ldg(p + i);
            o[2 * i] = make_float2(v.x, v.y);
            o[2 * i + 1] = make_float2(v.z, v.w);
        }
    }
}

// 8 activations (4 pairs) of batch row b at column k0 from the fp32 copy a.xf
__device__ __forceinline__ void load_xf8(const GemvArgs& a, int b, int64_t k0, float2 (&o)[4]) {
    const float4* p = reinterpret_cast<const float4*>(a.xf + b * a.K + k0);
    const float4 v0 = __ldg(p), v1 = __ldg(p + 1);
    o[0] = make_float2(v0.x, v0.y);
    o[1] = make_float2(v0.z, v0.w);
    o[2] = make_float2(v1.x, v1.y);
    o[3] = make_float2(v1.z, v1.w);
}

// NW words of quantized activations of batch row b starting at column k0
template <int NW>
__device__ __forceinline__ void load_xq(const GemvArgs& a, int b, int64_t k0, uint32_t (&o)[NW]) {
    if (NW == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.xq + b * a.K + k0));
        o[0] = v.x;
        o[NW - 1] = v.y;
        return;
    }
    const uint4* p = reinterpret_cast<const uint4*>(a.xq + b * a.K + k0);
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = __ldg(p + i);
        o[4 * i] = v.x;
        o[4 * i + 1] = v.y;
        o[4 * i + 2] = v.z;
        o[4 * i + 3] = v.w;
    }
}

// four code bytes -> two fp32 pairs of (code - off), exact
__device__ __forceinline__ void code_pairs(uint32_t c, float off, float2& p01, float2& p23) {
    const float2 neg = make_float2(-off, -off);
    p01 = fadd2(make_float2(byte_as_magic_float<0>(c), byte_as_magic_float<1>(c)), neg);
    p23 = fadd2(make_float2(byte_as_magic_float<2>(c), byte_as_magic_float<3>(c)), neg);
}

__device__ __forceinline__ float dot16(const float2 (&w)[8], const float2 (&x)[8]) {
    // two independent chains of four
    float2 s0 = ffma2(w[0], x[0], make_float2(0.0f, 0.0f));
    float2 s1 = ffma2(w[1], x[1], make_float2(0.0f, 0.0f));
#pragma unroll
    for (int k = 2; k < 8; k += 2) {
        s0 = ffma2(w[k], x[k], s0);
        s1 = ffma2(w[k + 1], x[k + 1], s1);
    }
    const float2 s = fadd2(s0, s1);
    return s.x + s.y;
}

__device__ __forceinline__ float dot8(const float2 (&w)[4], const float2 (&x)[4]) {
    float2 s = ffma2(w[0], x[0], make_float2(0.0f, 0.0f));
    s = ffma2(w[1], x[1], s);
    s = ffma2(w[2], x[2], s);
    s = ffma2(w[3], x[3], s);
    return s.x + s.y;
}

// (a & 0x0F0F0F0F) | (b & 0xF0F0F0F0): a nibble word merged with a word
// whose bits 4..5 of each byte hold the high code bits and bits 6..7 are 0
__device__ __forceinline__ uint32_t merge_nib(uint32_t a, uint32_t b) {
    return (a & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
}

// the 2-bit field k of every qh byte, moved to bits 4..5 (bits 6..7 zero)
template <int K>
__device__ __forceinline__ uint32_t qh_field(uint32_t h) {
    if (K == 0) return (h & 0x03030303u) << 4;
    if (K == 1) return (h & 0x0C0C0C0Cu) << 2;
    if (K == 2) return h & 0x30303030u;
    return (h >> 2) & 0x30303030u;
}

__device__ __forceinline__ float q6k_scale(uint32_t blk, int g, float d) {
    return d * static_cast<float>(lds_s8(blk + 192 + g));
}

// ------------------------------------------------------------ q6_K, wide
// lane = (block i = lane/4 of the chunk, q = lane%4). Lane q owns the groups
// q, q+4, q+8, q+12 (16 weights each): they share the 16 qh bytes
// [16q, 16q+16) (2-bit fields 0..3), and pairwise the ql bytes [16q, +16)
// (groups q, q+8: low / high nibbles) and [64+16q, +16) (groups q+4, q+12).
// Run s = 0 handles groups q and q+8, run s = 1 groups q+4 and q+12.
template <bool Q8, int NB, int R>
__device__ __forceinline__ void chunk_q6k_wide(const GemvArgs& a, uint32_t slot, int64_t row0,
                                               int64_t kb0, int ncb, int lane,
                                               float (&acc)[R][NB]) {
    constexpr int SEG = seg_stride<FMT_Q6_K>();
    const int i = lane >> 2, q = lane & 3;
    if (i >= ncb) return;
    const int64_t kb = kb0 + i;
    uint32_t blk[R];
    float ds[R][4];
    uint32_t hq[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        blk[r] = 0;
        ds[r][0] = ds[r][1] = ds[r][2] = ds[r][3] = 0.0f;
        hq[r][0] = hq[r][1] = hq[r][2] = hq[r][3] = 0u;
        if (row0 + r < a.N) {
            const int64_t st = ((row0 + r) * a.nb + kb0) * 210;
            blk[r] = slot + r * SEG + static_cast<uint32_t>(st & 15) + i * 210;
            const float d = half_bits_to_float(lds_u16(blk[r] + 208));
#pragma unroll
            for (int j = 0; j < 4; ++j) ds[r][j] = q6k_scale(blk[r], q + 4 * j, d);
            lds_words_unaligned<4>(blk[r] + 128 + 16 * q, hq[r]);
        }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int64_t kl = kb * 256 + 16 * (q + 4 * s);  // low-nibble group column
        const int64_t kh = kl + 128;                     // high-nibble group column
        float2 xl[Q8 ? 1 : NB][8], xh[Q8 ? 1 : NB][8];
        uint32_t xlq[Q8 ? NB : 1][4], xhq[Q8 ? NB : 1][4];
        int il0[Q8 ? NB : 1], ih0[Q8 ? NB : 1];
        float fl[Q8 ? NB : 1], fh[Q8 ? NB : 1];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= a.B) break;
            if (Q8) {
                load_xq<4>(a, b, kl, xlq[b]);
                load_xq<4>(a, b, kh, xhq[b]);
                int s0 = 0, s1 = 0;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    s0 = __dp4a(static_cast<int>(xlq[b][m]), 0x01010101, s0);
                    s1 = __dp4a(static_cast<int>(xhq[b][m]), 0x01010101, s1);
                }
                il0[b] = kMagicI - 32 * s0;
                ih0[b] = kMagicI - 32 * s1;
                fl[b] = __ldg(a.xs + b * (a.K / 32) + kl / 32);
                fh[b] = __ldg(a.xs + b * (a.K / 32) + kh / 32);
            } else {
                load_x16(a, b, kl, xl[b]);
                load_x16(a, b, kh, xh[b]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= a.N) break;
            uint32_t qlw[4];
            lds_words_unaligned<4>(blk[r] + 16 * q + 64 * s, qlw);
            uint32_t cl[4], ch[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t h = hq[r][m];
                cl[m] = merge_nib(qlw[m], s == 0 ? qh_field<0>(h) : qh_field<1>(h));
                ch[m] = merge_nib(qlw[m] >> 4, s == 0 ? qh_field<2>(h) : qh_field<3>(h));
            }
            if (Q8) {
                const float2 dsr = make_float2(ds[r][s], ds[r][2 + s]);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b >= a.B) break;
                    int il = il0[b], ih = ih0[b];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        il = __dp4a(static_cast<int>(cl[m]), static_cast<int>(xlq[b][m]), il);
                        ih = __dp4a(static_cast<int>(ch[m]), static_cast<int>(xhq[b][m]), ih);
                    }
                    // exact integer partials as floats, times d*sc, times s_x
                    const float2 I = fadd2(make_float2(__int_as_float(il), __int_as_float(ih)),
                                           make_float2(-kMagicIF, -kMagicIF));
                    const float2 u = fmul2(I, dsr);
                    acc[r][b] = fmaf(u.x, fl[b], acc[r][b]);
                    acc[r][b] = fmaf(u.y, fh[b], acc[r][b]);
                }
            } else {
                float2 wl[8], wh[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    code_pairs(cl[m], kMagic + 32.0f, wl[2 * m], wl[2 * m + 1]);
                    code_pairs(ch[m], kMagic + 32.0f, wh[2 * m], wh[2 * m + 1]);
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b >= a.B) break;
                    acc[r][b] = fmaf(ds[r][s], dot16(wl, xl[b]), acc[r][b]);
                    acc[r][b] = fmaf(ds[r][2 + s], dot16(wh, xh[b]), acc[r][b]);
                }
            }
        }
    }
}

// ------------------------------------------------------------ q6_K, narrow
// One block per pass: lane l decodes weights 8l..8l+7 (group l/2): ql bytes
// (8l mod 128)..+8 (nibble 4*(l/16)), qh bytes (8l mod 64)..+8 (field l/8).
template <bool Q8, int NB, int R>
__device__ __forceinline__ void chunk_q6k_narrow(const GemvArgs& a, uint32_t slot, int64_t row0,
                                                 int64_t kb0, int ncb, int lane,
                                                 float (&acc)[R][NB]) {
    constexpr int SEG = seg_stride<FMT_Q6_K>();
    const uint32_t nib_sh = 4u * static_cast<uint32_t>(lane >> 4);
    const uint32_t qh_sh = 2u * static_cast<uint32_t>(lane >> 3);
    uint32_t lead[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        lead[r] = static_cast<uint32_t>((((row0 + r) * a.nb + kb0) * 210) & 15);
    for (int i = 0; i < ncb; ++i) {
        const int64_t k0 = (kb0 + i) * 256 + 8 * lane;
        uint32_t c[R][2];
        float ds[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            c[r][0] = c[r][1] = 0u;
            ds[r] = 0.0f;
            if (row0 + r < a.N) {
                const uint32_t blk = slot + r * SEG + lead[r] + i * 210;
                uint32_t lw[2], hw[2];
                lds_words_unaligned<2>(blk + ((8 * lane) & 127), lw);
                lds_words_unaligned<2>(blk + 128 + ((8 * lane) & 63), hw);
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    c[r][m] = ((lw[m] >> nib_sh) & 0x0F0F0F0Fu) |
                              (((hw[m] >> qh_sh) & 0x03030303u) << 4);
                ds[r] = q6k_scale(blk, lane >> 1, half_bits_to_float(lds_u16(blk + 208)));
            }
        }
        if (Q8) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                uint32_t xw[2];
                load_xq<2>(a, b, k0, xw);
                const int sx = __dp4a(static_cast<int>(xw[1]), 0x01010101,
                                      __dp4a(static_cast<int>(xw[0]), 0x01010101, 0));
                const float f = __ldg(a.xs + b * (a.K / 32) + k0 / 32);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    int I = kMagicI - 32 * sx;
                    I = __dp4a(static_cast<int>(c[r][0]), static_cast<int>(xw[0]), I);
                    I = __dp4a(static_cast<int>(c[r][1]), static_cast<int>(xw[1]), I);
                    acc[r][b] = fmaf((__int_as_float(I) - kMagicIF) * ds[r], f, acc[r][b]);
                }
            }
        } else {
            float2 w[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                code_pairs(c[r][0], kMagic + 32.0f, w[r][0], w[r][1]);
                code_pairs(c[r][1], kMagic + 32.0f, w[r][2], w[r][3]);
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                float2 x[4];
                load_xf8(a, b, k0, x);
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r][b] = fmaf(ds[r], dot8(w[r], x), acc[r][b]);
            }
        }
    }
}

// ------------------------------------------------------------ Q4_0 / Q8_0
// codes c[m], m < 8, hold the elements 4m..4m+3 of a 32-element block in
// byte order (Q4_0: low nibbles of qs are elements 0..15, high 16..31).
template <int FMT>
__device__ __forceinline__ void q32_codes(uint32_t blk, uint32_t (&c)[8]) {
    if (FMT == FMT_Q4_0) {
        uint32_t qw[4];
        lds_words_unaligned<4>(blk + 2, qw);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            c[m] = qw[m] & 0x0F0F0F0Fu;
            c[4 + m] = (qw[m] >> 4) & 0x0F0F0F0Fu;
        }
    } else {
        lds_words_unaligned<8>(blk + 2, c);
    }
}

template <int FMT>
__device__ __forceinline__ void q32_pairs(const uint32_t* c, int n, float2* w) {
#pragma unroll
    for (int m = 0; m < n; ++m) {
        if (FMT == FMT_Q4_0)
            code_pairs(c[m], kMagic + 8.0f, w[2 * m], w[2 * m + 1]);
        else  // signed bytes: flip the sign bit to read 128 + q
            code_pairs(c[m] ^ 0x80808080u, kMagic + 128.0f, w[2 * m], w[2 * m + 1]);
    }
}

__device__ __forceinline__ float dot32(const float2 (&w)[16], const float2 (&x)[16]) {
    float2 s0 = make_float2(0.0f, 0.0f), s1 = s0, s2 = s0, s3 = s0;
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        s0 = ffma2(w[k], x[k], s0);
        s1 = ffma2(w[k + 1], x[k + 1], s1);
        s2 = ffma2(w[k + 2], x[k + 2], s2);
        s3 = ffma2(w[k + 3], x[k + 3], s3);
    }
    const float2 s = fadd2(fadd2(s0, s1), fadd2(s2, s3));
    return s.x + s.y;
}

// WIDE: lane = block i of the chunk (32 weights). The activations of the
// lane's block come in xv (chunk_x32), so that a caller can load them before
// it waits for the weights and use them for several matrices.
template <int NB>
__device__ __forceinline__ void chunk_x32(const GemvArgs& a, int64_t kb0, int ncb, int lane,
                                          float2 (&xv)[NB][16]) {
    if (lane >= ncb) return;
    const int64_t k0 = (kb0 + lane) * 32;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b >= a.B) break;
        float2 t0[8], t1[8];
        load_x16(a, b, k0, t0);
        load_x16(a, b, k0 + 16, t1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            xv[b][k] = t0[k];
            xv[b][8 + k] = t1[k];
        }
    }
}

// pulls the lane's activations of the chunk at kb0 into L1 (a hint)
template <int NB>
__device__ __forceinline__ void chunk_x32_prefetch(const GemvArgs& a, int64_t kb0, int ncb, int lane) {
    if (lane >= ncb) return;
    const int64_t k0 = (kb0 + lane) * 32;
    const int es = a.x_bf16 ? 2 : 4;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b >= a.B) break;
        const uint8_t* p = static_cast<const uint8_t*>(a.x) + (b * a.K + k0) * es;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
        if (es == 4) asm volatile("prefetch.global.L1 [%0];" ::"l"(p + 64));
    }
}

template <int FMT, int NB, int R>
__device__ __forceinline__ void chunk_q32_wide(const GemvArgs& a, uint32_t slot, int64_t row0,
                                               int64_t kb0, int ncb, int lane,
                                               const float2 (&xv)[NB][16], float (&acc)[R][NB]) {
    constexpr int BB = Fmt<FMT>::BB;
    constexpr int SEG = seg_stride<FMT>();
    const int i = lane;
    if (i >= ncb) return;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (row0 + r >= a.N) break;
        const int64_t st = ((row0 + r) * a.nb + kb0) * BB;
        const uint32_t blk = slot + r * SEG + static_cast<uint32_t>(st & 15) + i * BB;
        const float d = half_bits_to_float(lds_u16(blk));
        uint32_t c[8];
        q32_codes<FMT>(blk, c);
        float2 w[16];
        q32_pairs<FMT>(c, 8, w);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= a.B) break;
            acc[r][b] = fmaf(d, dot32(w, xv[b]), acc[r][b]);
        }
    }
}

// NARROW: 8 blocks per pass, lane = (block i = lane/4, quarter p = lane%4):
// weights 8p..8p+7 of the block (Q4_0: qs bytes 8*(p%2).., nibble p/2;
// Q8_0: qs bytes 8p..), so the warp's activations are 256 consecutive columns.
template <int FMT, bool Q8, int NB, int R>
__device__ __forceinline__ void chunk_q32_narrow(const GemvArgs& a, uint32_t slot, int64_t row0,
                                                 int64_t kb0, int ncb, int lane,
                                                 float (&acc)[R][NB]) {
    constexpr int BB = Fmt<FMT>::BB;
    constexpr int SEG = seg_stride<FMT>();
    const int p = lane & 3;
    uint32_t lead[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        lead[r] = static_cast<uint32_t>((((row0 + r) * a.nb + kb0) * BB) & 15);
    for (int pass = 0; pass * 8 < ncb; ++pass) {
        const int bi = pass * 8 + (lane >> 2);
        if (bi >= ncb) continue;
        const int64_t k0 = (kb0 + bi) * 32 + 8 * p;
        uint32_t c[R][2];
        float d[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            c[r][0] = c[r][1] = 0u;
            d[r] = 0.0f;
            if (row0 + r < a.N) {
                const uint32_t blk = slot + r * SEG + lead[r] + bi * BB;
                d[r] = half_bits_to_float(lds_u16(blk));
                uint32_t qw[2];
                if (FMT == FMT_Q4_0) {
                    lds_words_unaligned<2>(blk + 2 + 8 * (p & 1), qw);
                    const uint32_t sh = 4u * static_cast<uint32_t>(p >> 1);
                    c[r][0] = (qw[0] >> sh) & 0x0F0F0F0Fu;
                    c[r][1] = (qw[1] >> sh) & 0x0F0F0F0Fu;
                } else {
                    lds_words_unaligned<2>(blk + 2 + 8 * p, qw);
                    c[r][0] = qw[0];
                    c[r][1] = qw[1];
                }
            }
        }
        if (Q8) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                uint32_t xw[2];
                load_xq<2>(a, b, k0, xw);
                const int sx = __dp4a(static_cast<int>(xw[1]), 0x01010101,
                                      __dp4a(static_cast<int>(xw[0]), 0x01010101, 0));
                const float f = __ldg(a.xs + b * (a.K / 32) + k0 / 32);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    int I = (FMT == FMT_Q4_0) ? kMagicI - 8 * sx : kMagicI;
                    I = __dp4a(static_cast<int>(c[r][0]), static_cast<int>(xw[0]), I);
                    I = __dp4a(static_cast<int>(c[r][1]), static_cast<int>(xw[1]), I);
                    acc[r][b] = fmaf((__int_as_float(I) - kMagicIF) * d[r], f, acc[r][b]);
                }
            }
        } else {
            float2 w[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) q32_pairs<FMT>(c[r], 2, w[r]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                float2 x[4];
                load_xf8(a, b, k0, x);
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r][b] = fmaf(d[r], dot8(w[r], x), acc[r][b]);
            }
        }
    }
}

}  // namespace qmm
