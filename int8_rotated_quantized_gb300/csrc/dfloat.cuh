// Double-float arithmetic on the fp32 pipes (a value is hi + lo, two fp32
// numbers, |lo| <= half a step of hi after normalisation, about 48 significant
// bits).  Sums use Knuth's error-free two-sum, products Dekker's exact product
// through a fused multiply-add.  This GPU executes fp64 at a small fraction of
// its fp32 rate, so the kernels that need more than fp32 use these instead.
#pragma once

namespace convrot {

// s + e = a + b exactly, s = fl(a + b) (Knuth).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// s + e = a + b exactly for |a| >= |b| (Dekker).
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// (ah + al) + (bh + bl)
__device__ __forceinline__ void df_add(float ah, float al, float bh, float bl, float &rh, float &rl) {
    float s, e;
    two_sum(ah, bh, s, e);
    e = __fadd_rn(e, __fadd_rn(al, bl));
    fast_two_sum(s, e, rh, rl);
}

// (ah + al) * (bh + bl)
__device__ __forceinline__ void df_mul(float ah, float al, float bh, float bl, float &rh, float &rl) {
    const float p = __fmul_rn(ah, bh);
    float e = __fmaf_rn(ah, bh, -p);  // exact low part of ah * bh
    e = __fmaf_rn(ah, bl, __fmaf_rn(al, bh, e));
    fast_two_sum(p, e, rh, rl);
}

}  // namespace convrot
