// gemv.cu -- fused dequantize + matvec for q6_K / Q4_0 / Q8_0 weights
// (batch 1..16), the per-32 activation quantizer, the split-K reduction and
// the W_exp plane build.
//
// Why this shape (quantprobe "LAWS.md", Law 4 amendment L-15 / L-16): decode
// speed is set by bytes streamed AND by the format's unpack instruction cost.
// So the weights are streamed once, with 1-D bulk TMA copies into a
// per-warp ring of shared-memory slots (many bytes in flight, no per-thread
// load instructions), and the unpack is done with word-wide bit operations
// (4 codes per instruction) plus one byte-permute per code to form the
// float, instead of per-element shifts.
//
// q6_K element expansion ("57 - r54 MINFER_MMQ_Q6K_EXP" section 2.1): every
// 16-element group reads 16 consecutive ql bytes and 16 consecutive qh bytes
// with one shift pair; the code is (ql >> qsh & 0xF) | (qh >> qh_shift & 3) << 4.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <utility>

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

constexpr float kMagic = 8388608.0f;  // 2^23

// ------------------------------------------------------------ activations

// N consecutive activations of batch row b starting at column k0 (k0 a
// multiple of 8), as fp32.
template <int N>
__device__ __forceinline__ void load_x_run(const GemvArgs& a, int b, int64_t k0, float (&o)[N]) {
    if (a.x_bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                        b * a.K + k0);
#pragma unroll
        for (int i = 0; i < N / 8; ++i) {
            const uint4 v = __ldg(p + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                o[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) +
                                                          b * a.K + k0);
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 v = __ldg(p + i);
            o[4 * i] = v.x;
            o[4 * i + 1] = v.y;
            o[4 * i + 2] = v.z;
            o[4 * i + 3] = v.w;
        }
    }
}

// NW words of quantized activations of batch row b starting at column k0
template <int NW>
__device__ __forceinline__ void load_xq_run(const GemvArgs& a, int b, int64_t k0,
                                            uint32_t (&o)[NW]) {
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

// ------------------------------------------------------------ q6_K chunk
// lane = (block i = lane/4 of the chunk, quarter p = lane%4). Quarter p owns
// ql bytes [32p, 32p+32): elements 32p+t (low nibbles, qh bits 2*(p/2)) and
// 128+32p+t (high nibbles, qh bits 4+2*(p/2)), t < 32, with the qh bytes
// [32*(p%2), +32). It runs them as two half-steps of 16+16 elements.
template <bool Q8, int NB, int R>
__device__ __forceinline__ void chunk_q6k(const GemvArgs& a, uint32_t slot, int64_t row0,
                                          int64_t kb0, int ncb, int lane, float (&acc)[R][NB]) {
    constexpr int SEG = seg_stride<FMT_Q6_K>();
    const int i = lane >> 2, p = lane & 3;
    if (i >= ncb) return;
    const int64_t kb = kb0 + i;
    const uint32_t shl_lo = 4u - 2u * (p >> 1);
    const uint32_t shr_hi = 2u * (p >> 1);
#pragma unroll
    for (int hs = 0; hs < 2; ++hs) {
        const int64_t kl = kb * 256 + 32 * p + 16 * hs;  // low run column
        const int64_t kh = kl + 128;                     // high run column
        constexpr bool HOIST = (R > 1);
        float xl[HOIST ? NB : 1][16], xh[HOIST ? NB : 1][16];
        uint32_t ql8[HOIST ? NB : 1][4], qh8[HOIST ? NB : 1][4];
        int sxl[HOIST ? NB : 1], sxh[HOIST ? NB : 1];
        float sl_[HOIST ? NB : 1], sh_[HOIST ? NB : 1];
        if (HOIST) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                if (Q8) {
                    load_xq_run<4>(a, b, kl, ql8[b]);
                    load_xq_run<4>(a, b, kh, qh8[b]);
                    int s0 = 0, s1 = 0;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        s0 = __dp4a(static_cast<int>(ql8[b][m]), 0x01010101, s0);
                        s1 = __dp4a(static_cast<int>(qh8[b][m]), 0x01010101, s1);
                    }
                    sxl[b] = s0;
                    sxh[b] = s1;
                    sl_[b] = __ldg(a.xs + b * (a.K / 32) + kl / 32);
                    sh_[b] = __ldg(a.xs + b * (a.K / 32) + kh / 32);
                } else {
                    load_x_run<16>(a, b, kl, xl[b]);
                    load_x_run<16>(a, b, kh, xh[b]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r;
            if (row >= a.N) break;
            const int64_t st = (row * a.nb + kb0) * 210;
            const uint32_t blk = slot + r * SEG + static_cast<uint32_t>(st & 15) + i * 210;
            uint32_t qlw[4], qhw[4];
            lds_words_unaligned<4>(blk + 32 * p + 16 * hs, qlw);
            lds_words_unaligned<4>(blk + 128 + 32 * (p & 1) + 16 * hs, qhw);
            const float d = half_bits_to_float(lds_u16(blk + 208));
            const float dsl = d * static_cast<float>(lds_s8(blk + 192 + 2 * p + hs));
            const float dsh = d * static_cast<float>(lds_s8(blk + 200 + 2 * p + hs));
            uint32_t cl[4], ch[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                cl[m] = (qlw[m] & 0x0F0F0F0Fu) | ((qhw[m] << shl_lo) & 0x30303030u);
                ch[m] = ((qlw[m] >> 4) & 0x0F0F0F0Fu) | ((qhw[m] >> shr_hi) & 0x30303030u);
            }
            if (Q8) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b >= a.B) break;
                    uint32_t xlq[4], xhq[4];
                    int s0, s1;
                    float fl, fh;
                    if (HOIST) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            xlq[m] = ql8[b][m];
                            xhq[m] = qh8[b][m];
                        }
                        s0 = sxl[b];
                        s1 = sxh[b];
                        fl = sl_[b];
                        fh = sh_[b];
                    } else {
                        load_xq_run<4>(a, b, kl, xlq);
                        load_xq_run<4>(a, b, kh, xhq);
                        s0 = 0;
                        s1 = 0;
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            s0 = __dp4a(static_cast<int>(xlq[m]), 0x01010101, s0);
                            s1 = __dp4a(static_cast<int>(xhq[m]), 0x01010101, s1);
                        }
                        fl = __ldg(a.xs + b * (a.K / 32) + kl / 32);
                        fh = __ldg(a.xs + b * (a.K / 32) + kh / 32);
                    }
                    int il = 0, ih = 0;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        il = __dp4a(static_cast<int>(cl[m]), static_cast<int>(xlq[m]), il);
                        ih = __dp4a(static_cast<int>(ch[m]), static_cast<int>(xhq[m]), ih);
                    }
                    il -= 32 * s0;
                    ih -= 32 * s1;
                    acc[r][b] = fmaf(static_cast<float>(il) * dsl, fl, acc[r][b]);
                    acc[r][b] = fmaf(static_cast<float>(ih) * dsh, fh, acc[r][b]);
                }
            } else {
                float wl[16], wh[16];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    wl[4 * m + 0] = byte_as_magic_float<0>(cl[m]) - (kMagic + 32.0f);
                    wl[4 * m + 1] = byte_as_magic_float<1>(cl[m]) - (kMagic + 32.0f);
                    wl[4 * m + 2] = byte_as_magic_float<2>(cl[m]) - (kMagic + 32.0f);
                    wl[4 * m + 3] = byte_as_magic_float<3>(cl[m]) - (kMagic + 32.0f);
                    wh[4 * m + 0] = byte_as_magic_float<0>(ch[m]) - (kMagic + 32.0f);
                    wh[4 * m + 1] = byte_as_magic_float<1>(ch[m]) - (kMagic + 32.0f);
                    wh[4 * m + 2] = byte_as_magic_float<2>(ch[m]) - (kMagic + 32.0f);
                    wh[4 * m + 3] = byte_as_magic_float<3>(ch[m]) - (kMagic + 32.0f);
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b >= a.B) break;
                    float xa[16], xb[16];
                    if (HOIST) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            xa[t] = xl[b][t];
                            xb[t] = xh[b][t];
                        }
                    } else {
                        load_x_run<16>(a, b, kl, xa);
                        load_x_run<16>(a, b, kh, xb);
                    }
                    float sl = 0.0f, sh = 0.0f;
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        sl = fmaf(wl[t], xa[t], sl);
                        sh = fmaf(wh[t], xb[t], sh);
                    }
                    acc[r][b] = fmaf(dsl, sl, acc[r][b]);
                    acc[r][b] = fmaf(dsh, sh, acc[r][b]);
                }
            }
        }
    }
}

// ------------------------------------------------------------ Q4_0 / Q8_0 chunk
// lane = block i of the chunk (32 elements each).
template <int FMT, bool Q8, int NB, int R>
__device__ __forceinline__ void chunk_q32(const GemvArgs& a, uint32_t slot, int64_t row0,
                                          int64_t kb0, int ncb, int lane, float (&acc)[R][NB]) {
    constexpr int BB = Fmt<FMT>::BB;
    constexpr int SEG = seg_stride<FMT>();
    constexpr int NW = (FMT == FMT_Q4_0) ? 4 : 8;  // code words per block
    const int i = lane;
    if (i >= ncb) return;
    const int64_t kb = kb0 + i;
    const int64_t k0 = kb * 32;
    constexpr bool HOIST = (R > 1);
    float xv[HOIST ? NB : 1][32];
    uint32_t xq8[HOIST ? NB : 1][8];
    int sx[HOIST ? NB : 1];
    float sf[HOIST ? NB : 1];
    if (HOIST) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= a.B) break;
            if (Q8) {
                load_xq_run<8>(a, b, k0, xq8[b]);
                int s = 0;
#pragma unroll
                for (int m = 0; m < 8; ++m) s = __dp4a(static_cast<int>(xq8[b][m]), 0x01010101, s);
                sx[b] = s;
                sf[b] = __ldg(a.xs + b * (a.K / 32) + kb);
            } else {
                load_x_run<32>(a, b, k0, xv[b]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        if (row >= a.N) break;
        const int64_t st = (row * a.nb + kb0) * BB;
        const uint32_t blk = slot + r * SEG + static_cast<uint32_t>(st & 15) + i * BB;
        const float d = half_bits_to_float(lds_u16(blk));
        uint32_t qw[NW];
        lds_words_unaligned<NW>(blk + 2, qw);
        // codes in element order: c[0..3] elements 0..15, c[4..7] elements 16..31
        uint32_t c[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            if (FMT == FMT_Q4_0) {
                c[m] = qw[m] & 0x0F0F0F0Fu;
                c[4 + m] = (qw[m] >> 4) & 0x0F0F0F0Fu;
            } else {
                c[m] = qw[m];
                c[4 + m] = qw[4 + m];
            }
        }
        if (Q8) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                uint32_t xw[8];
                int s;
                float f;
                if (HOIST) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) xw[m] = xq8[b][m];
                    s = sx[b];
                    f = sf[b];
                } else {
                    load_xq_run<8>(a, b, k0, xw);
                    s = 0;
#pragma unroll
                    for (int m = 0; m < 8; ++m) s = __dp4a(static_cast<int>(xw[m]), 0x01010101, s);
                    f = __ldg(a.xs + b * (a.K / 32) + kb);
                }
                int I = 0;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    I = __dp4a(static_cast<int>(c[m]), static_cast<int>(xw[m]), I);
                if (FMT == FMT_Q4_0) I -= 8 * s;
                acc[r][b] = fmaf(static_cast<float>(I) * d, f, acc[r][b]);
            }
        } else {
            // code byte -> float: Q4_0 unsigned with offset 8, Q8_0 signed
            // (flip the sign bit to make it 128 + q).
            float w[32];
            constexpr float off = (FMT == FMT_Q4_0) ? (kMagic + 8.0f) : (kMagic + 128.0f);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t cw = (FMT == FMT_Q4_0) ? c[m] : (c[m] ^ 0x80808080u);
                w[4 * m + 0] = byte_as_magic_float<0>(cw) - off;
                w[4 * m + 1] = byte_as_magic_float<1>(cw) - off;
                w[4 * m + 2] = byte_as_magic_float<2>(cw) - off;
                w[4 * m + 3] = byte_as_magic_float<3>(cw) - off;
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) break;
                float xx[32];
                if (HOIST) {
#pragma unroll
                    for (int t = 0; t < 32; ++t) xx[t] = xv[b][t];
                } else {
                    load_x_run<32>(a, b, k0, xx);
                }
                float s = 0.0f;
#pragma unroll
                for (int t = 0; t < 32; ++t) s = fmaf(w[t], xx[t], s);
                acc[r][b] = fmaf(d, s, acc[r][b]);
            }
        }
    }
}

// ------------------------------------------------------------ the kernel

struct ItemCursor {
    int64_t item;
    int c, c_end;
};

__device__ __forceinline__ void cursor_set(const GemvArgs& a, ItemCursor& cur, int64_t item) {
    cur.item = item;
    if (item < a.n_items) {
        const int s = static_cast<int>(item % a.splits);
        cur.c = s * a.cps;
        cur.c_end = min(cur.c + a.cps, a.nchunks);
    }
}

template <int FMT, bool Q8, int NB, int R>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
    using F = Fmt<FMT>;
    constexpr int SEG = seg_stride<FMT>();
    constexpr int SLOT = SEG * R;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem) + warp * (kGemvSlots * SLOT);
    const uint32_t bars = smem_u32(smem) + kGemvWarps * kGemvSlots * SLOT + warp * kGemvSlots * 8;
    live_bump(a.st, a.live_slot);
    if (lane == 0) {
        for (int s = 0; s < kGemvSlots; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kGemvWarps + warp;
    const int64_t tw = static_cast<int64_t>(gridDim.x) * kGemvWarps;
    const int64_t tb16 = a.total_bytes & ~static_cast<int64_t>(15);

    // issue cursor: every lane tracks it, lane 0 performs the copies
    ItemCursor ic;
    cursor_set(a, ic, gw);
    uint32_t issued = 0;
    auto issue_next = [&]() {
        if (ic.item >= a.n_items) return;
        const uint32_t sidx = issued % kGemvSlots;
        const uint32_t dst = ring + sidx * SLOT;
        const uint32_t bar = bars + 8 * sidx;
        const int64_t row0 = (ic.item / a.splits) * R;
        const int64_t kb0 = static_cast<int64_t>(ic.c) * F::CB;
        const int64_t len = min(static_cast<int64_t>(F::CB), a.nb - kb0) * F::BB;
        if (lane == 0) {
            uint32_t total = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (row >= a.N) break;
                const int64_t st = (row * a.nb + kb0) * F::BB;
                const int64_t s16 = st & ~static_cast<int64_t>(15);
                const int64_t e16 = min((st + len + 15) & ~static_cast<int64_t>(15), tb16);
                if (e16 > s16) total += static_cast<uint32_t>(e16 - s16);
                // bytes past the last 16-byte boundary of W: plain loads
                for (int64_t q = max(e16, s16); q < st + len; ++q)
                    sts_u8(dst + r * SEG + static_cast<uint32_t>(q - s16), a.W[q]);
            }
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, total);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (row >= a.N) break;
                const int64_t st = (row * a.nb + kb0) * F::BB;
                const int64_t s16 = st & ~static_cast<int64_t>(15);
                const int64_t e16 = min((st + len + 15) & ~static_cast<int64_t>(15), tb16);
                if (e16 > s16)
                    bulk_g2s(dst + r * SEG, a.W + s16, static_cast<uint32_t>(e16 - s16), bar);
            }
        }
        ++issued;
        if (++ic.c >= ic.c_end) cursor_set(a, ic, ic.item + tw);
    };
    for (int s = 0; s < kGemvSlots; ++s) issue_next();

    uint32_t used = 0;
    for (int64_t item = gw; item < a.n_items; item += tw) {
        const int64_t row0 = (item / a.splits) * R;
        const int split = static_cast<int>(item % a.splits);
        const int c0 = split * a.cps, c1 = min(c0 + a.cps, a.nchunks);
        float acc[R][NB];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = 0.0f;
        for (int c = c0; c < c1; ++c) {
            const uint32_t sidx = used % kGemvSlots;
            if (!mbar_wait(bars + 8 * sidx, (used / kGemvSlots) & 1u)) {
                // give up: wait (bounded) for this warp's copies in flight, flag, leave
                for (uint32_t u = used + 1; u < issued; ++u)
                    (void)mbar_wait(bars + 8 * (u % kGemvSlots), (u / kGemvSlots) & 1u);
                if (lane == 0) atomicOr(a.st.err, DERR_GEMV_TIMEOUT);
                return;
            }
            const int64_t kb0 = static_cast<int64_t>(c) * F::CB;
            const int ncb = static_cast<int>(min(static_cast<int64_t>(F::CB), a.nb - kb0));
            const uint32_t slot = ring + sidx * SLOT;
            if (FMT == FMT_Q6_K)
                chunk_q6k<Q8, NB, R>(a, slot, row0, kb0, ncb, lane, acc);
            else
                chunk_q32<FMT, Q8, NB, R>(a, slot, row0, kb0, ncb, lane, acc);
            __syncwarp();
            ++used;
            issue_next();
        }
        // deterministic butterfly reduction, then one store per (row, batch)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float v = warp_sum(acc[r][b]);
                if (lane == ((r * NB + b) & 31) && row < a.N && b < a.B) {
                    if (a.splits == 1)
                        a.y[b * a.N + row] = v;
                    else
                        a.part[(static_cast<int64_t>(split) * a.B + b) * a.N + row] = v;
                }
            }
        }
    }
}

// ------------------------------------------------------------ dispatch

size_t gemv_smem_bytes(int fmt, int R) {
    int seg = fmt == FMT_Q6_K ? seg_stride<FMT_Q6_K>()
                              : (fmt == FMT_Q4_0 ? seg_stride<FMT_Q4_0>() : seg_stride<FMT_Q8_0>());
    return static_cast<size_t>(kGemvWarps) * kGemvSlots * seg * R + kGemvWarps * kGemvSlots * 8;
}

int gemv_chunk_blocks(int fmt) {
    return fmt == FMT_Q6_K ? Fmt<FMT_Q6_K>::CB : Fmt<FMT_Q4_0>::CB;
}

using GemvKernel = void (*)(const GemvArgs);

template <int FMT, bool Q8>
static GemvKernel pick(int NB, int R) {
    if (NB == 1 && R == 4) return gemv_kernel<FMT, Q8, 1, 4>;
    if (NB == 1 && R == 1) return gemv_kernel<FMT, Q8, 1, 1>;
    if (NB == 2 && R == 2) return gemv_kernel<FMT, Q8, 2, 2>;
    if (NB == 4 && R == 1) return gemv_kernel<FMT, Q8, 4, 1>;
    if (NB == 8 && R == 1) return gemv_kernel<FMT, Q8, 8, 1>;
    if (NB == 16 && R == 1) return gemv_kernel<FMT, Q8, 16, 1>;
    return nullptr;
}

static GemvKernel pick_kernel(int fmt, bool q8, int NB, int R) {
    switch (fmt) {
    case FMT_Q6_K: return q8 ? pick<FMT_Q6_K, true>(NB, R) : pick<FMT_Q6_K, false>(NB, R);
    case FMT_Q4_0: return q8 ? pick<FMT_Q4_0, true>(NB, R) : pick<FMT_Q4_0, false>(NB, R);
    case FMT_Q8_0: return q8 ? pick<FMT_Q8_0, true>(NB, R) : pick<FMT_Q8_0, false>(NB, R);
    }
    return nullptr;
}

// Sets the kernel's shared-memory opt-in and returns its resident CTAs per SM;
// both are computed once per (kernel, device) and cached.
int gemv_occupancy(int fmt, bool q8, int NB, int R) {
    GemvKernel k = pick_kernel(fmt, q8, NB, R);
    if (!k) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    static std::mutex mu;
    static std::map<std::pair<int, GemvKernel>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, k});
    if (it != cache.end()) return it->second;
    const size_t smem = gemv_smem_bytes(fmt, R);
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kGemvThreads, smem) != cudaSuccess)
        n = 0;
    cache[{dev, k}] = n;
    return n;
}

cudaError_t gemv_launch(int fmt, bool q8, int NB, int R, int grid, cudaStream_t s,
                        const GemvArgs& a) {
    GemvKernel k = pick_kernel(fmt, q8, NB, R);
    if (!k) return cudaErrorInvalidValue;
    const size_t smem = gemv_smem_bytes(fmt, R);
    // the shared-memory opt-in is set once per kernel (gemv_occupancy, called
    // by the planner before the first launch), so that a launch inside a
    // stream capture issues nothing but the launch itself
    if (gemv_occupancy(fmt, q8, NB, R) <= 0) return cudaErrorInvalidConfiguration;
    k<<<grid, kGemvThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------ split-K reduce

__global__ void splitk_reduce_kernel(const float* __restrict__ part, float* __restrict__ y,
                                     int splits, int64_t count, DevState st) {
    live_bump(st, 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v = 0.0f;
        for (int s = 0; s < splits; ++s) v += part[s * count + i];
        y[i] = v;
    }
}

cudaError_t splitk_reduce_launch(const float* part, float* y, int splits, int64_t count,
                                 cudaStream_t s, DevState st) {
    const int threads = 256;
    int64_t blocks = (count + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    splitk_reduce_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(part, y, splits, count, st);
    return cudaGetLastError();
}

// ------------------------------------------------------------ q8 quantizer
// One thread per 32-element block: amax, s = amax / 127 (IEEE fp32 division),
// x_q = round-half-even(x / s) clamped to [-127, 127]. A block whose scale is
// zero quantizes to zeros.

__device__ __forceinline__ void a16_store(uint16_t* a16, int64_t K, int64_t r, int64_t kb,
                                          const int (&q)[32]);

__global__ void quantize_q8_kernel(const void* __restrict__ x, int x_bf16, int64_t rows,
                                   int64_t K, int8_t* __restrict__ xq, float* __restrict__ xs,
                                   uint16_t* __restrict__ a16, int64_t rows_pad, DevState st) {
    live_bump(st, 3);
    const int64_t nkb = K / 32;
    const int64_t nblk = rows_pad * nkb;
    for (int64_t blk = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; blk < nblk;
         blk += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = blk / nkb, kb = blk % nkb;
        int q[32];
        if (r < rows) {
            float v[32];
            if (x_bf16) {
                const uint4* p = reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(x) + r * K + kb * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 u = __ldg(p + i);
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                        v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                    }
                }
            } else {
                const float4* p =
                    reinterpret_cast<const float4*>(static_cast<const float*>(x) + r * K + kb * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 u = __ldg(p + i);
                    v[4 * i] = u.x;
                    v[4 * i + 1] = u.y;
                    v[4 * i + 2] = u.z;
                    v[4 * i + 3] = u.w;
                }
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
            const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                int t = 0;
                if (s != 0.0f) {
                    t = __float2int_rn(__fdiv_rn(v[i], s));
                    t = max(-127, min(127, t));
                }
                q[i] = t;
            }
            if (xq) {
                uint32_t pk[8];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    pk[m] = (q[4 * m] & 0xFF) | ((q[4 * m + 1] & 0xFF) << 8) |
                            ((q[4 * m + 2] & 0xFF) << 16) | ((q[4 * m + 3] & 0xFF) << 24);
                uint4* o = reinterpret_cast<uint4*>(xq + r * K + kb * 32);
                o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            xs[r * nkb + kb] = s;
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = 0;
        }
        if (a16) a16_store(a16, K, r, kb, q);
    }
}

// GEMM A-operand tile layout (must match gemm.cu): for every 128-row tile mt
// and every 32-column block kb, one 8 KB tile of fp16 values laid out as
// core matrices [row group rg (16)][k group kc (4)][row (8)][8 values].
__device__ __forceinline__ void a16_store(uint16_t* a16, int64_t K, int64_t r, int64_t kb,
                                          const int (&q)[32]) {
    const int64_t nkb = K / 32;
    const int64_t mt = r >> 7;
    const int rr = static_cast<int>(r & 127);
    uint16_t* tile = a16 + (mt * nkb + kb) * (128 * 32);
    const int rg = rr >> 3, rw = rr & 7;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = __half_as_ushort(__int2half_rn(q[8 * kc + 2 * j]));
            const uint32_t hi = __half_as_ushort(__int2half_rn(q[8 * kc + 2 * j + 1]));
            h[j] = lo | (hi << 16);
        }
        uint4* o = reinterpret_cast<uint4*>(tile + (rg * 4 + kc) * 64 + rw * 8);
        *o = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

cudaError_t quantize_q8_launch(const void* x, int x_bf16, int64_t rows, int64_t K, int8_t* xq,
                               float* xs, uint16_t* a16, cudaStream_t s, DevState st) {
    const int64_t rows_pad = a16 ? ((rows + 127) / 128) * 128 : rows;
    const int threads = 256;
    int64_t blocks = (rows_pad * (K / 32) + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    quantize_q8_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(x, x_bf16, rows, K, xq, xs,
                                                                    a16, rows_pad, st);
    return cudaGetLastError();
}

// ------------------------------------------------------------ W_exp plane
// plane[n][k] = q(n,k) - 32, one thread per 16-element group (16 ql bytes,
// 16 qh bytes, one shift pair), "57 - r54 MINFER_MMQ_Q6K_EXP" section 2.2.

__global__ void plane_build_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t K,
                                   int8_t* __restrict__ plane, DevState st) {
    live_bump(st, 4);
    const int64_t ngr = K / 16;
    const int64_t total = N * ngr;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = g / ngr, j = g % ngr;
        const int64_t sb = j / 16;
        const int e0 = static_cast<int>(j % 16) * 16;
        const uint8_t* blk = W + (n * (K / 256) + sb) * 210;
        const int s1 = 4 * (e0 >> 7), s2 = 2 * (e0 >> 6);
        uint32_t out[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t w = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int e = e0 + 4 * m + t;
                const int lo = (blk[e & 127] >> s1) & 0xF;
                const int hi = (blk[128 + (e & 63)] >> s2) & 0x3;
                w |= static_cast<uint32_t>(((lo | (hi << 4)) - 32) & 0xFF) << (8 * t);
            }
            out[m] = w;
        }
        *reinterpret_cast<uint4*>(plane + n * K + sb * 256 + e0) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

cudaError_t plane_build_launch(const uint8_t* W, int64_t N, int64_t K, int8_t* plane,
                               cudaStream_t s, DevState st) {
    const int threads = 256;
    int64_t blocks = (N * (K / 16) + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    plane_build_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(W, N, K, plane, st);
    return cudaGetLastError();
}

}  // namespace qmm
