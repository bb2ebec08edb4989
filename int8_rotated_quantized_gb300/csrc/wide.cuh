// Helpers of the row-wise kernels that hold 32 consecutive elements per
// thread: 256-bit global accesses, the in-register Walsh-Hadamard transform,
// the row maximum and the rounding of codes.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "fwht.cuh"

namespace convrot {

__device__ __forceinline__ void ld256(const void *p, uint32_t *r) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
}

__device__ __forceinline__ void st256(void *p, const uint32_t *r) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]),
                 "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Walsh-Hadamard butterflies on blocks of 2^LOGB elements, 32 consecutive
// elements per thread, blocks wider than 32 spread over 2^LOGB / 32
// consecutive lanes.  (a, c) -> (a + c, a - c) on indices k and k ^ h gives the
// Sylvester order H[i][j] = (-1)^popcount(i & j).
template <int LOGB>
__device__ __forceinline__ void fwht32(float (&e)[32], int lane) {
    constexpr int B = 1 << LOGB;
    constexpr int HMAX = B < 32 ? B : 32;
    if constexpr (HMAX > 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const float a = e[i], c = e[i + 1];
            e[i] = a + c;
            e[i + 1] = a - c;
        }
    }
#pragma unroll
    for (int h = 2; h < HMAX; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            if ((i & h) == 0) addsub2(e[i], e[i + 1], e[i + h], e[i + h + 1]);
    }
    constexpr int L = B / 32;
#pragma unroll
    for (int m = 1; m < L; m <<= 1) {
        const float sg = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int i0 = 0; i0 < 32; i0 += 8) {
            float p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(0xffffffffu, e[i0 + i], m);
#pragma unroll
            for (int i = 0; i < 8; i += 2) sfma2(sg, e[i0 + i], e[i0 + i + 1], p[i], p[i + 1]);
        }
    }
}

__device__ __forceinline__ void unpack_bf16x32(const uint32_t (&w)[16], float (&e)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        e[2 * i] = __uint_as_float(w[i] << 16);
        e[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 32 codes rne(e * inv) as fp16 values (64 bytes).
__device__ __forceinline__ void store_codes32(float (&e)[32], float inv, __half *dst) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) mul2c(e[i], e[i + 1], inv);
#pragma unroll
    for (int i = 0; i < 32; i += 2) add2c(e[i], e[i + 1], kMagicF16);
    const __half2 k1152 = __half2half2(__ushort_as_half((unsigned short)0x6480));
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t v = __byte_perm(__float_as_uint(e[2 * i]), __float_as_uint(e[2 * i + 1]), 0x5410);
        __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&v), k1152);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    st256(dst, w);
    st256(dst + 16, w + 8);
}

// 32 codes rne(e * inv) as int8 (32 bytes).
__device__ __forceinline__ void store_codes32(float (&e)[32], float inv, int8_t *dst) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) mul2c(e[i], e[i + 1], inv);
#pragma unroll
    for (int i = 0; i < 32; i += 2) add2c(e[i], e[i + 1], kMagicI8);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t lo = __byte_perm(__float_as_uint(e[4 * k]), __float_as_uint(e[4 * k + 1]), 0x0040);
        const uint32_t hi = __byte_perm(__float_as_uint(e[4 * k + 2]), __float_as_uint(e[4 * k + 3]), 0x0040);
        w[k] = __byte_perm(lo, hi, 0x5410);
    }
    st256(dst, w);
}

__device__ __forceinline__ float amax32(const float (&e)[32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(e[i]), fabsf(e[i + 8]));
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], fmaxf(fabsf(e[i + 16]), fabsf(e[i + 24])));
    return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// int8 x 4 -> four fp32 values of the same integers: bias each byte by 128
// (xor 0x80), splice it under the exponent of 2^23 (0x4B000000, where the fp32
// spacing is 1), and subtract 2^23 + 128 exactly.
__device__ __forceinline__ void codes_to_f32x4(uint32_t w, float *e) {
    const uint32_t x = w ^ 0x80808080u;
    e[0] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540));
    e[1] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541));
    e[2] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542));
    e[3] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543));
    add2c(e[0], e[1], -8388736.0f);
    add2c(e[2], e[3], -8388736.0f);
}

// int8 x 4 -> two fp16x2 words holding the same integers: bias each byte by
// 128 (xor 0x80), splice it under the fp16 exponent of 1024 (0x64), and
// subtract 1152 = 1024 + 128 exactly.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(x), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(x), "r"(0x64646464u));
    const __half2 k = __half2half2(__ushort_as_half((unsigned short)0x6480));
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), k);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), k);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
}

}  // namespace convrot
