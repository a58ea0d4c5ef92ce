// quant.cuh -- the per-32 activation quantizer shared by the kernels that
// quantize activations: s = amax / 127 (IEEE fp32 division), x_q =
// round-half-even(x / s) clamped to [-127, 127]; a block whose scale is zero
// quantizes to zeros (quantprobe "LAWS.md", Law 4 amendment L-15: int8
// activations for the dp4a-style integer dot products).
#pragma once

#include <stdint.h>

namespace qmm {

// 32 activations of row r, block kb, from fp32 or bf16 [rows][K]
__device__ __forceinline__ void load_x32(const void* x, int x_bf16, int64_t K, int64_t r,
                                         int64_t kb, float (&v)[32]) {
    if (x_bf16) {
        const uint4* p =
            reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + r * K + kb * 32);
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
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + r * K + kb * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 u = __ldg(p + i);
            v[4 * i] = u.x;
            v[4 * i + 1] = u.y;
            v[4 * i + 2] = u.z;
            v[4 * i + 3] = u.w;
        }
    }
}

// quantizes one block; returns its scale s
__device__ __forceinline__ float quantize_block32(const float (&v)[32], int (&q)[32]) {
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
    return s;
}

}  // namespace qmm
