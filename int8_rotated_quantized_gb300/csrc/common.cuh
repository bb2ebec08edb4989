// Shared device helpers of libconvrot (CUDA, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace convrot {

// Bits of the sticky device error word.
enum : unsigned {
    DEVERR_INDEX = 1u,    // an embedding id outside [0, V)
    DEVERR_TIMEOUT = 2u,  // a pipeline wait exceeded its limit
};

// Wall-clock limit of one pipeline wait (ns).  Legitimate waits last
// microseconds; the limit only turns a would-be hang into an error.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) {
    return __uint_as_float(h16 << 16);
}

__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return float_to_bf16_bits(lo) | (float_to_bf16_bits(hi) << 16);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Checked builds (-DCONVROT_CHECKED, the library variant libconvrot_checked):
// CR_IN_BOUNDS(cond) guards a global-memory access with the condition that its
// index lies inside the logical tensor; a false condition records a failure
// in this translation unit's device flag (reported by convrot_get_error as
// CONVROT_ERR_BOUNDS) and the access is skipped.  Release builds compile the
// condition away.
#ifdef CONVROT_CHECKED
void register_bounds_flag(unsigned (*read_and_clear)());
static __device__ unsigned g_bounds_fail;
#define CR_IN_BOUNDS(cond) ((cond) ? true : (atomicOr(&::convrot::g_bounds_fail, 1u), false))
namespace {
struct BoundsFlagRegistration {
    BoundsFlagRegistration() { register_bounds_flag(&read_and_clear); }
    static unsigned read_and_clear() {
        unsigned v = 0;
        if (cudaMemcpyFromSymbol(&v, g_bounds_fail, sizeof v) != cudaSuccess) return 0u;
        if (v != 0u) {
            const unsigned zero = 0u;
            (void)cudaMemcpyToSymbol(g_bounds_fail, &zero, sizeof zero);
        }
        return v;
    }
};
static BoundsFlagRegistration g_bounds_registration;
}  // namespace
#else
#define CR_IN_BOUNDS(cond) true
#endif
// An access of `len` elements at element offset `off` of a buffer holding
// `extent` elements.
#define CR_SPAN(off, len, extent) \
    CR_IN_BOUNDS((int64_t)(off) >= 0 && (int64_t)(off) + (int64_t)(len) <= (int64_t)(extent))

}  // namespace convrot
