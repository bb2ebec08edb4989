// Measurement entry for a roofline denominator: the dense int8 rate of this
// GPU's tensor cores through the only int8 MMA it offers, the warp-level
// mma.sync (tcgen05 has no int8 kind on sm_103a).  The kernel issues nothing
// but independent m16n8k32 s8 x s8 -> s32 MMAs from every warp of a grid of
// four 256-thread CTAs per SM; the caller times it and divides the operation
// count by the time.
#include "convrot.h"
#include "internal.h"
#include "launch_cache.h"

namespace convrot {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 4;
constexpr int kChains = 8;  // independent accumulators per warp

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kProbeThreads) mma_s8_rate_kernel(int iters, int32_t *sink) {
    const uint32_t t = threadIdx.x;
    const uint32_t a0 = t * 0x01010101u, a1 = a0 ^ 0x5a5a5a5au, a2 = a0 ^ 0x33333333u, a3 = a0 ^ 0x0f0f0f0fu;
    const uint32_t b0 = (t + 7u) * 0x01010101u, b1 = b0 ^ 0x3c3c3c3cu;
    int acc[kChains][4];
#pragma unroll
    for (int j = 0; j < kChains; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) mma_s8_16832(acc[j], a0, a1, a2, a3, b0, b1);
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
    // one value per CTA keeps the MMAs live
    for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    __shared__ int red[kProbeThreads / 32];
    if ((t & 31) == 0) red[t >> 5] = s;
    __syncthreads();
    if (t == 0) {
        int v = 0;
        for (int w = 0; w < kProbeThreads / 32; ++w) v += red[w];
        sink[blockIdx.x] = v;
    }
}

}  // namespace
}  // namespace convrot

extern "C" {

int convrot_probe_mma_s8_rate(int iters, int32_t *sink, size_t sink_bytes, double *ops, convrot_stream_t stream) {
    if (iters <= 0 || sink == nullptr || ops == nullptr || ((uintptr_t)sink & 3u)) return CONVROT_ERR_INVALID_ARG;
    using namespace convrot;
    const int grid = sm_count() * kProbeCtasPerSm;
    if (grid <= 0) return CONVROT_ERR_CUDA;
    if (sink_bytes < (size_t)grid * sizeof(int32_t)) return CONVROT_ERR_INVALID_ARG;
    // 2 * 16 * 8 * 32 operations per MMA, kChains MMAs per warp per iteration
    *ops = 2.0 * 16 * 8 * 32 * (double)kChains * (double)iters * (double)(kProbeThreads / 32) * (double)grid;
    mma_s8_rate_kernel<<<grid, kProbeThreads, 0, (cudaStream_t)stream>>>(iters, sink);
    return cudaGetLastError() == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}

}  // extern "C"
