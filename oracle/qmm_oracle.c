/*
 * qmm_oracle.c -- plain, slow CPU reference for matrix multiplication against
 * block-quantized weights (q6_K, Q4_0, Q8_0, and the K-quant ladder formats
 * Q4_K and Q2_K).
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this file. The CUDA library never does:
 * the two share no code, header, table or constant. The numbering of formats
 * and activation kinds below is written out again here on purpose.
 *
 * Everything follows the plain definition of each quantity, with no blocking,
 * fusion or reordering beyond what the definition states:
 *   - each weight is decoded from its block exactly (the decoded value is an
 *     exact fp32 number, see orc_weight),
 *   - dot products accumulate in double precision in increasing k,
 *   - the activation quantizer takes its rounding decisions in fp32, the
 *     precision the quantized format itself is defined in (fp32 scale).
 *
 * Sources (page title, then section):
 *   [MINFER]  "57 - r54 MINFER_MMQ_Q6K_EXP: an exit valve for the 1.52 GB
 *             W_exp plane", section 2.1 (the q6_K element expansion
 *             v = ((ql>>qsh)&0xF) | (((qh>>qh_shift)&3)<<4) - 32 done per
 *             16-element group) and section 2.2 (the W_exp plane: one
 *             centered int8 byte per weight, od x id bytes).
 *   [LAWS]    quantprobe "LAWS.md", Law 4 amendment L-15 (matvec with dp4a
 *             on quantized activations).
 *   [X100]    "Chasing x100", "Where the wall actually fell: inversion"
 *             (routed experts kept resident and decoded in place; top-k
 *             routed expert FFN per token).
 *   [CBK]     "Chasing x100", "The kernel is ready" (a 2-bit and a 3-bit
 *             additive codebook matvec, checked against a bit-faithful CPU
 *             reference).
 *   [L16]     quantprobe "LAWS.md", Law 4, the per-format eta paragraph and
 *             amendment L-16 (metadata application density: Q2_K applies a
 *             scale and a min every 16 weights = 4 bytes at 2 bits, Q4_K
 *             every 32 weights = 16 bytes at 4 bits).
 *
 * Readings where the pages are silent (they print no byte order for the
 * nibbles): q6_K element i of a 256-weight super-block takes its low four
 * bits from ql[i mod 128] (low nibble for i < 128, high nibble otherwise),
 * its high two bits from qh[i mod 64] at bit 2*(i div 64), and its scale from
 * scales[i div 16]; every 16-element group therefore reads 16 consecutive ql
 * bytes and 16 consecutive qh bytes with one shift pair, as [MINFER] 2.1
 * describes the in-kernel expansion.
 *
 * The K-quant ladder formats ([L16]): the pages give their sub-block sizes
 * and that each sub-block carries a scale and a min, but no byte layout. The
 * reading here (the common K-quant super-block of 256 weights), weight =
 * d * scale_j * q - dmin * min_j for sub-block j:
 *   Q4_K, 144 bytes: d (fp16) | dmin (fp16) | 12 bytes holding eight 6-bit
 *     scales and eight 6-bit mins | 128 bytes of 4-bit codes. Sub-block j
 *     (32 weights) for j < 4: scale = b[j] & 63, min = b[j + 4] & 63; for
 *     j >= 4: scale = (b[j + 4] & 15) | (b[j - 4] >> 6) << 4, min =
 *     (b[j + 4] >> 4) | (b[j] >> 6) << 4, b the 12 bytes. Element i is nibble
 *     (i / 32) % 2 (0 = low) of code byte 32 * (i / 64) + i % 32.
 *   Q2_K, 84 bytes: 16 bytes (sub-block j = i / 16: low nibble scale, high
 *     nibble min) | 64 bytes of 2-bit codes | d (fp16) | dmin (fp16).
 *     Element i is the 2-bit field at bit 2 * ((i % 128) / 32) of code byte
 *     32 * (i / 128) + i % 32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* formats, numbered as the library's C interface numbers them */
#define ORC_Q4_0 1
#define ORC_Q8_0 2
#define ORC_Q6_K 3
#define ORC_Q4_K 4
#define ORC_Q2_K 5

/* activation element kinds */
#define ORC_X_F32 0
#define ORC_X_BF16 1

/* ------------------------------------------------------------------ */
/* scalar decoders                                                     */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16 -> double, exact for every finite input (subnormals
 * included: many q6_K scales d = fp16(|N(0,1)| * 2e-4) are subnormal). */
double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* 0.m * 2^-14 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 */
double orc_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_x(const void* x, int xkind, int64_t i) {
    if (xkind == ORC_X_BF16)
        return orc_bf16_to_double(((const uint16_t*)x)[i]);
    return (double)((const float*)x)[i];
}

/* ------------------------------------------------------------------ */
/* block formats                                                       */
/* ------------------------------------------------------------------ */

int orc_block_elems(int fmt) {
    switch (fmt) {
    case ORC_Q4_0: return 32;
    case ORC_Q8_0: return 32;
    case ORC_Q6_K: return 256;
    case ORC_Q4_K: return 256;
    case ORC_Q2_K: return 256;
    }
    return 0;
}

int orc_block_bytes(int fmt) {
    switch (fmt) {
    case ORC_Q4_0: return 2 + 16;              /* d fp16, 16 bytes of nibbles  */
    case ORC_Q8_0: return 2 + 32;              /* d fp16, 32 int8 values       */
    case ORC_Q6_K: return 128 + 64 + 16 + 2;   /* ql, qh, scales, d = 210 B    */
    case ORC_Q4_K: return 2 + 2 + 12 + 128;    /* d, dmin, scales+mins, codes  */
    case ORC_Q2_K: return 16 + 64 + 2 + 2;     /* scales+mins, codes, d, dmin  */
    }
    return 0;
}

/* size of the integer group that carries one weight-side scale factor */
int orc_group_elems(int fmt) { return fmt == ORC_Q6_K ? 16 : 32; }

/* q6_K: the unsigned 6-bit code of element i (0..255) of a super-block,
 * [MINFER] 2.1: low four bits from ql, high two bits from qh. */
int orc_q6k_code(const uint8_t* blk, int i) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    int lo = (ql[i % 128] >> (4 * (i / 128))) & 0xF;
    int hi = (qh[i % 64] >> (2 * (i / 64))) & 0x3;
    return lo | (hi << 4);
}

/* K-quant ladder formats (readings in the file header) */
static int is_kquant(int fmt) { return fmt == ORC_Q4_K || fmt == ORC_Q2_K; }

/* the unsigned code of element i (0..255): Q4_K 0..15, Q2_K 0..3 */
int orc_kq_code(int fmt, const uint8_t* blk, int i) {
    if (fmt == ORC_Q4_K) {
        const uint8_t* qs = blk + 16;
        return (qs[32 * (i / 64) + i % 32] >> (4 * ((i / 32) % 2))) & 0xF;
    }
    const uint8_t* qs = blk + 16;
    return (qs[32 * (i / 128) + i % 32] >> (2 * ((i % 128) / 32))) & 0x3;
}

/* the scale and the min of sub-block j (Q4_K: j < 8, Q2_K: j < 16) */
void orc_kq_scale_min(int fmt, const uint8_t* blk, int j, int* scale, int* min) {
    if (fmt == ORC_Q4_K) {
        const uint8_t* b = blk + 4;
        if (j < 4) {
            *scale = b[j] & 63;
            *min = b[j + 4] & 63;
        } else {
            *scale = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);
            *min = (b[j + 4] >> 4) | ((b[j] >> 6) << 4);
        }
        return;
    }
    *scale = blk[j] & 15;
    *min = blk[j] >> 4;
}

int orc_kq_sub_elems(int fmt) { return fmt == ORC_Q4_K ? 32 : 16; }

/* d and dmin of a K-quant super-block */
double orc_kq_d(int fmt, const uint8_t* blk) {
    int off = fmt == ORC_Q4_K ? 0 : 80;
    return orc_half_to_double((uint16_t)(blk[off] | (blk[off + 1] << 8)));
}
double orc_kq_dmin(int fmt, const uint8_t* blk) {
    int off = fmt == ORC_Q4_K ? 2 : 82;
    return orc_half_to_double((uint16_t)(blk[off] | (blk[off + 1] << 8)));
}

/* the two terms of a K-quant weight: d * scale * q and dmin * min, each an
 * exact double (11-bit d times at most 10 bits, 11-bit dmin times 6 bits) */
static void kq_terms(int fmt, const uint8_t* blk, int i, double* pos, double* neg) {
    int sc, mn;
    orc_kq_scale_min(fmt, blk, i / orc_kq_sub_elems(fmt), &sc, &mn);
    *pos = orc_kq_d(fmt, blk) * (double)(sc * orc_kq_code(fmt, blk, i));
    *neg = orc_kq_dmin(fmt, blk) * (double)mn;
}

/* integer value of element i before the weight-side scale: q6_K gives
 * sc[i/16] * (q - 32), Q4_0 gives q - 8, Q8_0 gives q. */
static int int_value(int fmt, const uint8_t* blk, int i) {
    if (fmt == ORC_Q6_K) {
        int sc = (int8_t)blk[192 + i / 16];
        return sc * (orc_q6k_code(blk, i) - 32);
    }
    if (fmt == ORC_Q4_0) {
        const uint8_t* qs = blk + 2;
        int q = (qs[i % 16] >> (4 * (i / 16))) & 0xF;
        return q - 8;
    }
    /* Q8_0 */
    return (int8_t)blk[2 + i];
}

/* the centered code without the sub-block scale (what the integer dot
 * products multiply): q6_K q-32, Q4_0 q-8, Q8_0 q */
int orc_centered_code(int fmt, const uint8_t* blk, int i) {
    if (fmt == ORC_Q6_K) return orc_q6k_code(blk, i) - 32;
    return int_value(fmt, blk, i);
}

/* the per-block fp16 scale d */
double orc_block_d(int fmt, const uint8_t* blk) {
    int off = (fmt == ORC_Q6_K) ? 208 : 0;
    uint16_t h = (uint16_t)(blk[off] | (blk[off + 1] << 8));
    return orc_half_to_double(h);
}

/* the sub-block scale that multiplies group g: q6_K scales[g], else 1 */
int orc_group_scale(int fmt, const uint8_t* blk, int g) {
    if (fmt == ORC_Q6_K) return (int8_t)blk[192 + g];
    return 1;
}

/* Dequantized weight k of a row: d * (integer value). d has an 11-bit
 * significand and |integer value| <= 1024 needs at most 11 bits, so the
 * product is exact in fp32 as well as in double. */
double orc_weight(int fmt, const uint8_t* row, int64_t k) {
    int be = orc_block_elems(fmt);
    const uint8_t* blk = row + (k / be) * orc_block_bytes(fmt);
    if (is_kquant(fmt)) {
        double pos, neg;
        kq_terms(fmt, blk, (int)(k % be), &pos, &neg);
        return pos - neg;
    }
    return orc_block_d(fmt, blk) * (double)int_value(fmt, blk, (int)(k % be));
}

/* dequantize a whole row of K weights */
void orc_dequant_row(int fmt, const uint8_t* row, int64_t K, double* out) {
    for (int64_t k = 0; k < K; ++k) out[k] = orc_weight(fmt, row, k);
}

static const uint8_t* row_ptr(int fmt, const uint8_t* W, int64_t K, int64_t n) {
    return W + n * (K / orc_block_elems(fmt)) * orc_block_bytes(fmt);
}

/* ------------------------------------------------------------------ */
/* float-activation matvec: y[b][n] = sum_k w[n][k] * x[b][k]          */
/* ------------------------------------------------------------------ */

/* one dot product in double; *absum receives the scale the float tolerance
 * is stated against: sum_k |w*x|, and for the K-quant formats, whose weight
 * is the difference of two terms, sum_k (|d*scale*q| + |dmin*min|) * |x| */
double orc_dot_float(int fmt, const uint8_t* row, int64_t K, const void* x,
                     int xkind, int64_t xoff, double* absum) {
    double s = 0.0, a = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = load_x(x, xkind, xoff + k);
        double p = orc_weight(fmt, row, k) * xv;
        s += p;
        if (is_kquant(fmt)) {
            int be = orc_block_elems(fmt);
            double pos, neg;
            kq_terms(fmt, row + (k / be) * orc_block_bytes(fmt), (int)(k % be), &pos, &neg);
            a += (fabs(pos) + fabs(neg)) * fabs(xv);
        } else {
            a += fabs(p);
        }
    }
    if (absum) *absum = a;
    return s;
}

void orc_gemv_float(int fmt, const uint8_t* W, int64_t N, int64_t K,
                    const void* x, int xkind, int B, double* y, double* absum) {
    for (int b = 0; b < B; ++b)
        for (int64_t n = 0; n < N; ++n)
            y[b * N + n] = orc_dot_float(fmt, row_ptr(fmt, W, K, n), K, x, xkind,
                                         (int64_t)b * K, absum ? &absum[b * N + n] : NULL);
}

/* ------------------------------------------------------------------ */
/* activation quantizer: per 32-element block, s = amax/127 (fp32),     */
/* x_q = round-half-even(x / s) clamped to [-127, 127]; amax == 0 gives */
/* s = 0 and x_q = 0. Decisions taken in fp32. Reading: a block whose   */
/* scale amax/127 rounds to zero in fp32 (amax below about 9e-44) is     */
/* treated like the all-zero block, since x/s is undefined there.        */
/* ------------------------------------------------------------------ */

void orc_quantize_q8(const void* x, int xkind, int64_t rows, int64_t K,
                     int8_t* xq, float* s) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b0 = 0; b0 < K; b0 += 32) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float v = (float)load_x(x, xkind, r * K + b0 + i);
                float av = fabsf(v);
                if (av > amax) amax = av;
            }
            float sc = amax / 127.0f;
            s[r * (K / 32) + b0 / 32] = sc;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (sc != 0.0f) {
                    float v = (float)load_x(x, xkind, r * K + b0 + i);
                    float t = v / sc;
                    float rq = nearbyintf(t); /* default mode: to nearest, ties to even */
                    if (rq > 127.0f) rq = 127.0f;
                    if (rq < -127.0f) rq = -127.0f;
                    q = (int)rq;
                }
                xq[r * K + b0 + i] = (int8_t)q;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* quantized-activation matvec ([LAWS] L-15: integer dot products)      */
/* I_g = sum_{k in g} x_q[k] * c[k]   (c the centered code, exact int)  */
/* y   = sum_g s_x[block(g)] * d * sc_g * I_g                            */
/* ------------------------------------------------------------------ */

/* integer partial of group g (global group index along the row) */
int64_t orc_group_int(int fmt, const uint8_t* row, const int8_t* xq, int64_t g) {
    int be = orc_block_elems(fmt), ge = orc_group_elems(fmt);
    int64_t k0 = g * ge;
    const uint8_t* blk = row + (k0 / be) * orc_block_bytes(fmt);
    int64_t acc = 0;
    for (int i = 0; i < ge; ++i) {
        int e = (int)((k0 + i) % be);
        acc += (int64_t)xq[k0 + i] * orc_centered_code(fmt, blk, e);
    }
    return acc;
}

double orc_dot_q8(int fmt, const uint8_t* row, int64_t K, const int8_t* xq,
                  const float* s, double* absum) {
    int be = orc_block_elems(fmt), ge = orc_group_elems(fmt);
    double y = 0.0, a = 0.0;
    for (int64_t g = 0; g < K / ge; ++g) {
        int64_t k0 = g * ge;
        const uint8_t* blk = row + (k0 / be) * orc_block_bytes(fmt);
        double d = orc_block_d(fmt, blk);
        int sc = orc_group_scale(fmt, blk, (int)((k0 % be) / ge));
        double sx = (double)s[k0 / 32];
        int64_t I = orc_group_int(fmt, row, xq, g);
        y += sx * d * (double)sc * (double)I;
        if (absum)
            for (int i = 0; i < ge; ++i)
                a += fabs(orc_weight(fmt, row, k0 + i) * sx * (double)xq[k0 + i]);
    }
    if (absum) *absum = a;
    return y;
}

void orc_gemv_q8(int fmt, const uint8_t* W, int64_t N, int64_t K, const int8_t* xq,
                 const float* s, int B, double* y, double* absum) {
    for (int b = 0; b < B; ++b)
        for (int64_t n = 0; n < N; ++n)
            y[b * N + n] = orc_dot_q8(fmt, row_ptr(fmt, W, K, n), K, xq + (int64_t)b * K,
                                      s + (int64_t)b * (K / 32),
                                      absum ? &absum[b * N + n] : NULL);
}

/* Prefill GEMM, Y[m][n] = quantized-activation dot of X[m] with W[n], for a
 * list of (m, n) pairs (so that full-size matrices can be spot-checked).
 * xq/s are the quantized activations of all M rows. */
void orc_gemm_q8_pairs(int fmt, const uint8_t* W, int64_t K, const int8_t* xq,
                       const float* s, const int64_t* ms, const int64_t* ns,
                       int64_t count, double* y, double* absum) {
    for (int64_t i = 0; i < count; ++i)
        y[i] = orc_dot_q8(fmt, row_ptr(fmt, W, K, ns[i]), K, xq + ms[i] * K,
                          s + ms[i] * (K / 32), absum ? &absum[i] : NULL);
}

/* float-mode matvec for a list of (b, n) pairs */
void orc_gemv_float_pairs(int fmt, const uint8_t* W, int64_t K, const void* x,
                          int xkind, const int64_t* bs, const int64_t* ns,
                          int64_t count, double* y, double* absum) {
    for (int64_t i = 0; i < count; ++i)
        y[i] = orc_dot_float(fmt, row_ptr(fmt, W, K, ns[i]), K, x, xkind, bs[i] * K,
                             absum ? &absum[i] : NULL);
}

/* ------------------------------------------------------------------ */
/* W_exp plane ([MINFER] 2.2): one centered int8 per weight, row-major  */
/* N x K, plane[n][k] = q(n,k) - 32                                      */
/* ------------------------------------------------------------------ */

void orc_plane_q6k(const uint8_t* W, int64_t N, int64_t K, int8_t* plane) {
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = row_ptr(ORC_Q6_K, W, K, n);
        for (int64_t k = 0; k < K; ++k)
            plane[n * K + k] =
                (int8_t)(orc_q6k_code(row + (k / 256) * 210, (int)(k % 256)) - 32);
    }
}

/* ------------------------------------------------------------------ */
/* routed MoE ([X100] inversion section; top-k with softmax gates)      */
/* ------------------------------------------------------------------ */

/* top-k by logit value, ties to the lower expert index, then a softmax over
 * the k selected logits (renormalized over the selection), in double. */
void orc_route_topk_softmax(const float* logits, int T, int E, int k,
                            int32_t* idx, double* gate) {
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            idx[t * k + j] = best;
        }
        double mx = (double)l[idx[t * k]];
        double z = 0.0;
        for (int j = 0; j < k; ++j) z += exp((double)l[idx[t * k + j]] - mx);
        for (int j = 0; j < k; ++j) gate[t * k + j] = exp((double)l[idx[t * k + j]] - mx) / z;
    }
    free(taken);
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Routed expert FFN for T tokens, float activations:
 *   g = Wg_e x_t, u = Wu_e x_t, h = silu(g) * u, o = Wd_e h,
 *   y_t = sum_j gate[t][j] * o_{idx[t][j]}.
 * wg/wu hold I x H matrices, wd holds H x I matrices, one pointer per expert.
 * bound (optional, [T][H]) receives the float tolerance the GPU result is
 * held to: the per-matvec bound 1e-4 * sum|w x| + 1e-6 carried through
 * silu (|silu'| <= 1.1) and the down projection. h_out (optional,
 * [T][k][I]) receives h. */
void orc_moe_float(int fmt, int H, int I, const uint8_t* const* wg,
                   const uint8_t* const* wu, const uint8_t* const* wd, int T, int k,
                   const int32_t* idx, const double* gate, const void* x, int xkind,
                   double* y, double* bound, double* h_out) {
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* dh = (double*)malloc(sizeof(double) * (size_t)I);
    for (int t = 0; t < T; ++t) {
        for (int n = 0; n < H; ++n) {
            y[(int64_t)t * H + n] = 0.0;
            if (bound) bound[(int64_t)t * H + n] = 1e-6;
        }
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            double gw = gate[t * k + j];
            for (int i = 0; i < I; ++i) {
                double ag, au;
                double g = orc_dot_float(fmt, row_ptr(fmt, wg[e], H, i), H, x, xkind,
                                         (int64_t)t * H, &ag);
                double u = orc_dot_float(fmt, row_ptr(fmt, wu[e], H, i), H, x, xkind,
                                         (int64_t)t * H, &au);
                double sg = silu(g);
                h[i] = sg * u;
                double eg = 1e-4 * ag + 1e-6, eu = 1e-4 * au + 1e-6;
                dh[i] = fabs(u) * 1.1 * eg + (fabs(sg) + 1.1 * eg) * eu + 1e-6 * fabs(h[i]);
                if (h_out) h_out[((int64_t)t * k + j) * I + i] = h[i];
            }
            for (int n = 0; n < H; ++n) {
                const uint8_t* row = row_ptr(fmt, wd[e], I, n);
                double o = 0.0, a = 0.0, p = 0.0;
                for (int i = 0; i < I; ++i) {
                    double w = orc_weight(fmt, row, i);
                    o += w * h[i];
                    a += fabs(w * h[i]);
                    p += fabs(w) * dh[i];
                }
                y[(int64_t)t * H + n] += gw * o;
                if (bound) bound[(int64_t)t * H + n] += gw * (1e-4 * a + p);
            }
        }
    }
    free(h);
    free(dh);
}

/* ------------------------------------------------------------------ */
/* expert-grouped MoE prefill ([LAWS] L-30: prefill divides parameters, */
/* not bytes): the routed expert FFN of orc_moe_float with every matmul  */
/* on quantized activations, as the prefill GEMM computes it:            */
/*   g = W_g (q8 x), u = W_u (q8 x), h = silu(g) * u,                    */
/*   o = W_d (q8 h), y_t = sum_j gate[t][j] * o_{idx[t][j]}.             */
/* Reading: h is re-quantized per 32 like any GEMM input; its rounding   */
/* decisions are taken in fp32 on h rounded to fp32.                     */
/* ------------------------------------------------------------------ */

/* tight (optional, [T][H]): the bound that holds when every code of the
 * quantized h equals the oracle's: per expert output 1e-4 * sum|w_d h^| +
 * 1e-6, gate-weighted. loose (optional, [T][H]): a bound that holds for any
 * h within its propagated error of the oracle's (the GEMM bar 1e-4 *
 * sum|w x^| + 1e-6 on g and u, carried through silu with |silu'| <= 1.1):
 * every code may then be off by one step, so each h element adds
 * |w_d| * (s + dh + max dh / 254) to it (s its block's scale). */
void orc_moe_q8(int fmt, int H, int I, const uint8_t* const* wg, const uint8_t* const* wu,
                const uint8_t* const* wd, int T, int k, const int32_t* idx, const double* gate,
                const void* x, int xkind, double* y, double* tight, double* loose) {
    int8_t* xq = (int8_t*)malloc((size_t)H);
    float* sx = (float*)malloc(sizeof(float) * (size_t)(H / 32));
    float* hf = (float*)malloc(sizeof(float) * (size_t)I);
    int8_t* hq = (int8_t*)malloc((size_t)I);
    float* sh = (float*)malloc(sizeof(float) * (size_t)(I / 32));
    double* dh = (double*)malloc(sizeof(double) * (size_t)I);
    double* stepw = (double*)malloc(sizeof(double) * (size_t)I);
    for (int t = 0; t < T; ++t) {
        orc_quantize_q8((const uint8_t*)x + (size_t)t * H * (xkind == ORC_X_BF16 ? 2 : 4), xkind, 1, H, xq,
                        sx);
        for (int n = 0; n < H; ++n) {
            y[(int64_t)t * H + n] = 0.0;
            if (tight) tight[(int64_t)t * H + n] = 0.0;
            if (loose) loose[(int64_t)t * H + n] = 0.0;
        }
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            double gw = gate[t * k + j];
            for (int i = 0; i < I; ++i) {
                double ag, au;
                double g = orc_dot_q8(fmt, row_ptr(fmt, wg[e], H, i), H, xq, sx, &ag);
                double u = orc_dot_q8(fmt, row_ptr(fmt, wu[e], H, i), H, xq, sx, &au);
                double sg = silu(g);
                hf[i] = (float)(sg * u);
                double eg = 1e-4 * ag + 1e-6, eu = 1e-4 * au + 1e-6;
                dh[i] = fabs(u) * 1.1 * eg + (fabs(sg) + 1.1 * eg) * eu + 1e-6 * fabs(sg * u);
            }
            orc_quantize_q8(hf, ORC_X_F32, 1, I, hq, sh);
            for (int b = 0; b < I / 32; ++b) {
                double mx = 0.0;
                for (int i = 32 * b; i < 32 * b + 32; ++i)
                    if (dh[i] > mx) mx = dh[i];
                for (int i = 32 * b; i < 32 * b + 32; ++i) stepw[i] = (double)sh[b] + dh[i] + mx / 254.0;
            }
            for (int n = 0; n < H; ++n) {
                const uint8_t* row = row_ptr(fmt, wd[e], I, n);
                double ad;
                double o = orc_dot_q8(fmt, row, I, hq, sh, &ad);
                y[(int64_t)t * H + n] += gw * o;
                double tb = 1e-4 * ad + 1e-6;
                if (tight) tight[(int64_t)t * H + n] += gw * tb;
                if (loose) {
                    double p = 0.0;
                    for (int i = 0; i < I; ++i) p += fabs(orc_weight(fmt, row, i)) * stepw[i];
                    loose[(int64_t)t * H + n] += gw * (tb + 1e-4 * p + p);
                }
            }
        }
    }
    free(xq);
    free(sx);
    free(hf);
    free(hq);
    free(sh);
    free(dh);
    free(stepw);
}

/* ------------------------------------------------------------------ */
/* additive-codebook matrix ([CBK]). The pages give no layout; the one   */
/* read here: M (2 or 3) codebooks of 256 entries of 8 fp16 values,      */
/* books[m][c][j]; codes[n][g][m] one byte per codebook per group of 8   */
/* consecutive weights; an fp16 scale per row. Weight 8g + j of row n:   */
/*   w = scale[n] * sum_m books[m][codes[n][g][m]][j]                    */
/* (2 bits per weight for M = 2, 3 for M = 3, plus the shared books).    */
/* ------------------------------------------------------------------ */

/* the M terms of weight k of row n (each an exact double) */
static void cbk_terms(int M, const uint8_t* codes, const uint16_t* books, const uint16_t* scales,
                      int64_t K, int64_t n, int64_t k, double* t) {
    int64_t g = k / 8;
    int j = (int)(k % 8);
    double s = orc_half_to_double(scales[n]);
    for (int m = 0; m < M; ++m) {
        int c = codes[(n * (K / 8) + g) * M + m];
        t[m] = s * orc_half_to_double(books[((int64_t)m * 256 + c) * 8 + j]);
    }
}

double orc_cbk_weight(int M, const uint8_t* codes, const uint16_t* books, const uint16_t* scales, int64_t K,
                      int64_t n, int64_t k) {
    double t[3], w = 0.0;
    cbk_terms(M, codes, books, scales, K, n, k, t);
    for (int m = 0; m < M; ++m) w += t[m];
    return w;
}

/* y[b][n] = sum_k w[n][k] x[b][k] in double; absum the tolerance scale:
 * sum_k sum_m |term_m| |x| (the kernel sums the codebooks' terms apart) */
void orc_cbk_gemv(int M, const uint8_t* codes, const uint16_t* books, const uint16_t* scales, int64_t N,
                  int64_t K, const void* x, int xkind, int B, double* y, double* absum) {
    for (int b = 0; b < B; ++b)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, a = 0.0, t[3];
            for (int64_t k = 0; k < K; ++k) {
                double xv = load_x(x, xkind, (int64_t)b * K + k);
                cbk_terms(M, codes, books, scales, K, n, k, t);
                double w = 0.0;
                for (int m = 0; m < M; ++m) {
                    w += t[m];
                    a += fabs(t[m]) * fabs(xv);
                }
                acc += w * xv;
            }
            y[b * N + n] = acc;
            if (absum) absum[b * N + n] = a;
        }
}
