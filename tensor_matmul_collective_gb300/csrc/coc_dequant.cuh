// w8A16 dequantisation shared by the fused kernel's dequant warps
// (coc_kernel.cu) and the streaming pre-pass (coc_w8_prepass.cu), so both
// produce the same bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "coc_internal.h"

namespace coc {

// Scale / zero-point table geometry of one rank's weight.
struct W8Layout {
    int gran;    // COC_SCALE_TENSOR / CHANNEL / GROUP
    int group;   // rows of k per group (per-group tables)
    int n;       // columns
};

// Dequantisation constants of one dequant thread: its 8 consecutive columns
// j0..j0+7 of one rank's weight at one k-block, and the conversion of one
// 8-column row (two words of int8 q) to 8 dequantised 16-bit values,
//     Wd = rne( (q - z) * s ),
// exact up to the one rounding.  q - z is formed exactly with the published
// bias trick (Kim et al., "Who Says Elephants Can't Run", 2022): flipping the
// sign bits gives the byte u = q + 128; placed under a float's exponent
// pattern it reads as 2^p + u, and subtracting 2^p + 128 + z leaves q - z.
//   fp16:  under 0x64 (binary16 1024 + u), subtract 1152 + z (exact in
//          binary16: an integer below 2048), then one binary16 multiply.
//   bf16:  under 0x4B (binary32 2^23 + u), subtract 2^23 + 128 + z, multiply
//          by the widened bf16 scale (exact in binary32: <= 9 x 8 bits), then
//          one rounding to bf16.
// Columns past n get scale 0 (their products with the zero-filled A are 0).
template <bool BF16>
struct Dq;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Offset of the scale / zero-point table row for weight row `row` (per
// group: one table row per `group` rows of k; otherwise the single row).
__device__ __forceinline__ long long w8_table_row(const W8Layout& L, int row) {
    return (L.gran == COC_SCALE_GROUP) ? static_cast<long long>(row / L.group) * L.n : 0LL;
}

// The 8 zero points of columns j0..j0+7 (0 if none, or past n).
__device__ __forceinline__ void load_w8_zeros(const W8Layout& L, const int8_t* zp, int row, int j0, int (&z)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = 0;
    if (zp == nullptr) return;
    if (L.gran == COC_SCALE_TENSOR) {
        const int zv = zp[0];
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = zv;
    } else if (j0 + 8 <= L.n) {
        const uint2 z8 = __ldg(reinterpret_cast<const uint2*>(zp + w8_table_row(L, row) + j0));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            z[e] = static_cast<int8_t>((z8.x >> (8 * e)) & 0xFFu);
            z[4 + e] = static_cast<int8_t>((z8.y >> (8 * e)) & 0xFFu);
        }
    }
}

// The 8 scales of columns j0..j0+7 as four 32-bit words of two 16-bit values.
__device__ __forceinline__ void load_w8_scale_words(const W8Layout& L, const uint16_t* sc, int row, int j0, uint32_t (&w)[4]) {
    if (L.gran == COC_SCALE_TENSOR) {
        const uint32_t v = sc[0];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = v | (v << 16);
    } else if (j0 + 8 <= L.n) {
        const uint4 s8 = __ldg(reinterpret_cast<const uint4*>(sc + w8_table_row(L, row) + j0));
        w[0] = s8.x; w[1] = s8.y; w[2] = s8.z; w[3] = s8.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = 0u;
    }
}

template <>
struct Dq<false> {
    __half2 s[4], c[4];   // scales and 1152 + z, column pairs
    __device__ __forceinline__ void load(const W8Layout& L, const uint16_t* sc, const int8_t* zp, int row, int j0) {
        uint32_t w[4];
        load_w8_scale_words(L, sc, row, j0, w);
        int z[8];
        load_w8_zeros(L, zp, row, j0, z);
        set(w, z);
    }
    // from the 8 scales (four words of two) and the 8 zero points
    __device__ __forceinline__ void set(const uint32_t (&w)[4], const int (&z)[8]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[e] = *reinterpret_cast<const __half2*>(&w[e]);
            c[e] = __floats2half2_rn(static_cast<float>(1152 + z[2 * e]), static_cast<float>(1152 + z[2 * e + 1]));
        }
    }
    __device__ __forceinline__ uint4 convert(uint2 q8) const {
        const uint32_t qw[2] = {q8.x, q8.y};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t u = qw[h] ^ 0x80808080u;
            const uint32_t a = prmt(u, 0x64646464u, 0x4140u);   // binary16 1024 + u0, 1024 + u1
            const uint32_t b = prmt(u, 0x64646464u, 0x4342u);   // 1024 + u2, 1024 + u3
            const __half2 d0 = __hmul2_rn(__hsub2(*reinterpret_cast<const __half2*>(&a), c[2 * h]), s[2 * h]);
            const __half2 d1 = __hmul2_rn(__hsub2(*reinterpret_cast<const __half2*>(&b), c[2 * h + 1]), s[2 * h + 1]);
            o[2 * h] = *reinterpret_cast<const uint32_t*>(&d0);
            o[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&d1);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

template <>
struct Dq<true> {
    float s[8], c[8];     // widened scales and 2^23 + 128 + z
    __device__ __forceinline__ void load(const W8Layout& L, const uint16_t* sc, const int8_t* zp, int row, int j0) {
        uint32_t w[4];
        load_w8_scale_words(L, sc, row, j0, w);
        int z[8];
        load_w8_zeros(L, zp, row, j0, z);
        set(w, z);
    }
    // from the 8 scales (four words of two) and the 8 zero points
    __device__ __forceinline__ void set(const uint32_t (&w)[4], const int (&z)[8]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[2 * e] = __uint_as_float(w[e] << 16);
            s[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = 8388736.0f + static_cast<float>(z[e]);   // exact
    }
    __device__ __forceinline__ uint4 convert(uint2 q8) const {
        const uint32_t qw[2] = {q8.x, q8.y};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t u = qw[h] ^ 0x80808080u;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float f = __uint_as_float(prmt(u, 0x4B000000u, 0x7650u + e));   // 2^23 + u_e
                v[e] = __fmul_rn(__fsub_rn(f, c[4 * h + e]), s[4 * h + e]);
            }
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2], v[3]);
            o[2 * h] = *reinterpret_cast<const uint32_t*>(&b0);
            o[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&b1);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

}  // namespace coc
