// Packed fp32 helpers shared by the row-wise kernels (rotation butterflies and
// the rounding of codes).
#pragma once

#include <stdint.h>

namespace convrot {

// The same butterflies with two lanes of fp32 per instruction (f32x2, round
// to nearest per lane, so every value equals the scalar computation).

// (a, c) -> (a + c, a - c) on the pairs (a0, a1) and (c0, c1).
__device__ __forceinline__ void addsub2(float &a0, float &a1, float &c0, float &c1) {
    asm("{\n .reg .b64 ra, rc, rs, rd;\n mov.b64 ra, {%0, %1};\n mov.b64 rc, {%2, %3};\n"
        " add.rn.f32x2 rs, ra, rc;\n sub.rn.f32x2 rd, ra, rc;\n mov.b64 {%0, %1}, rs;\n mov.b64 {%2, %3}, rd;\n}"
        : "+f"(a0), "+f"(a1), "+f"(c0), "+f"(c1));
}

// (e0, e1) <- (s * e0 + p0, s * e1 + p1) with s = +-1: one rounding, equal to e + p or p - e.
__device__ __forceinline__ void sfma2(float s, float &e0, float &e1, float p0, float p1) {
    asm("{\n .reg .b64 rs, re, rp;\n mov.b64 rs, {%2, %2};\n mov.b64 re, {%0, %1};\n mov.b64 rp, {%3, %4};\n"
        " fma.rn.f32x2 re, rs, re, rp;\n mov.b64 {%0, %1}, re;\n}"
        : "+f"(e0), "+f"(e1)
        : "f"(s), "f"(p0), "f"(p1));
}

// (e0, e1) <- (e0 * k + c, e1 * k + c): one rounding per lane.
__device__ __forceinline__ void fma2c(float &e0, float &e1, float k, float c) {
    asm("{\n .reg .b64 rk, re, rc;\n mov.b64 rk, {%2, %2};\n mov.b64 re, {%0, %1};\n mov.b64 rc, {%3, %3};\n"
        " fma.rn.f32x2 re, re, rk, rc;\n mov.b64 {%0, %1}, re;\n}"
        : "+f"(e0), "+f"(e1)
        : "f"(k), "f"(c));
}

__device__ __forceinline__ void mul2c(float &e0, float &e1, float k) {
    asm("{\n .reg .b64 rk, re;\n mov.b64 rk, {%2, %2};\n mov.b64 re, {%0, %1};\n"
        " mul.rn.f32x2 re, re, rk;\n mov.b64 {%0, %1}, re;\n}"
        : "+f"(e0), "+f"(e1)
        : "f"(k));
}

// (a0, a1) <- (a0 * b0, a1 * b1), one rounding per lane.
__device__ __forceinline__ void mul2v(float &a0, float &a1, float b0, float b1) {
    asm("{\n .reg .b64 ra, rb;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
        " mul.rn.f32x2 ra, ra, rb;\n mov.b64 {%0, %1}, ra;\n}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

__device__ __forceinline__ void add2c(float &e0, float &e1, float c) {
    asm("{\n .reg .b64 rc, re;\n mov.b64 rc, {%2, %2};\n mov.b64 re, {%0, %1};\n"
        " add.rn.f32x2 re, re, rc;\n mov.b64 {%0, %1}, re;\n}"
        : "+f"(e0), "+f"(e1)
        : "f"(c));
}

// Codes are rne(u * inv) with |u * inv| < 127.5 (|u| <= amax_u and
// inv = fp32(127 / amax_u)), so the result already lies in [-127, 127].  The
// rounding is done by adding 1.5 * 2^23 (+ an offset): in [2^23, 2^24) the
// fp32 spacing is 1, so the sum is u * inv rounded to the nearest integer,
// ties to even, and the integer sits in the low mantissa bits.

constexpr float kMagicI8 = 12582912.0f;   // 1.5 * 2^23: low byte = two's-complement code
constexpr float kMagicF16 = 12608640.0f;  // 1.5 * 2^23 + 0x6480: low 16 bits = fp16 bits of 1152 + code

}  // namespace convrot
