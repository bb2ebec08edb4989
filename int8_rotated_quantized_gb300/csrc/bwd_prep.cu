// The transient bf16 weight of the default bf16 backward mode of a frozen
// ConvRot base (MOSS-Image LoRA training guide, section 4.1: the backward
// option takes bf16, the default, or int8; sd-scripts PR #2461, Summary:
// frozen base, grad_x only): W_eff^T = bf16((scale_w (.) Wq) R)^T, correctly
// rounded from a double-float value.  (The one-off int8 backward weight is in
// bwd_weight.cu.)
#include "common.cuh"
#include "dfloat.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "wide.cuh"

namespace convrot {
namespace {

// ------------------------------------------------- bf16-mode backward weight --

// The transient dequantization of the bf16 backward: WeffT[k][n] =
// bf16(scale_w[n] * (H_b q_n)[k] / sqrt(b)), correctly rounded from a
// double-float value.  A CTA takes 64 weight rows and one Hadamard block, so
// each output row segment it writes is 128 contiguous bytes.
constexpr int kDeqRows = 64;

// bf16 bits of hi + lo (|lo| <= ulp(hi) / 2), rounded to nearest even: hi
// decides unless its low 16 bits sit exactly on a bf16 tie, where the sign
// of lo (or, if lo is 0, evenness) breaks it.  Rounding up means increasing
// the magnitude, which is +1 on the sign-magnitude bits for either sign.
__device__ __forceinline__ uint16_t df_to_bf16(float hi, float lo) {
    const uint32_t u = __float_as_uint(hi);
    const uint32_t low = u & 0xffffu;
    const uint32_t r = u >> 16;
    bool up;
    if (low != 0x8000u)
        up = low > 0x8000u;
    else if (lo == 0.f)
        up = (r & 1u) != 0;
    else
        up = (lo > 0.f) == (hi > 0.f);
    return (uint16_t)(r + (up ? 1u : 0u));
}

// A CTA takes 64 weight rows and KT = max(128, B) columns; each thread owns
// 32 consecutive codes of one row (two 16-byte loads), turns them into exact
// fp32 values (byte splice), transforms them in registers (packed fp32
// butterflies, log2(B / 32) stages across lanes; integer sums below 2^15, so
// exact), rounds every value s * u / sqrt(B) to bf16 and writes it into a
// shared tile [KT][64] whose 8-column groups are xor-swizzled by the writer's
// 32-column chunk; the tile leaves as 16-byte stores (128-byte row segments of
// T).  (A persistent form of this kernel, loading the next tile's codes while
// transforming the current one, measured slower: 64-68 us against 58 us.)
//
// Rounding.  With (sh, sl) the row factor s / sqrt(B) as a double-float, the
// value is v = u (sh + sl).  The fp32 product p = u * sh differs from it by
// less than 2.5 fp32 steps of p (half a step from the product's rounding,
// under two from u * sl, since |sl| <= one step of sh), so the bf16 rounding
// of p is already the correct rounding of v unless p's low 16 bits lie within
// that distance of 0x8000, a bf16 rounding midpoint.  Groups of 8 values with
// such a p (about 1 in 900 per thread) are rounded again from the exact
// double-float value hi + lo; the rest keep the rounding of p.
template <int B>
__global__ void __launch_bounds__(512) dequant_t_kernel(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K,
                                                        float ch, float cl, uint16_t *T) {
    constexpr int KT = B > 128 ? B : 128;
    constexpr int TPR = KT / 32;  // threads per row
    constexpr int LOGB = B == 8 ? 3 : B == 16 ? 4 : B == 32 ? 5 : B == 64 ? 6 : B == 128 ? 7 : 8;
    __shared__ __align__(16) uint16_t dtile[KT * kDeqRows];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int rl = tid / TPR, c = tid - rl * TPR;
    const int64_t n0 = (int64_t)blockIdx.x * kDeqRows;
    const int64_t k0 = (int64_t)blockIdx.y * KT;
    const int64_t n = n0 + rl;
    const bool ok = n < N && k0 + 32 * c < K;
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    float s = 0.f;
    if (ok && CR_SPAN(n * K + k0 + 32 * c, 16, N * K)) {  // K is a multiple of 16: the second 16 codes may lie past the row
        const uint4 *src = reinterpret_cast<const uint4 *>(Wq + n * K + k0 + 32 * c);
        const uint4 v0 = __ldg(src);
        const uint4 v1 = k0 + 32 * c + 16 < K && CR_SPAN(n * K + k0 + 32 * c + 16, 16, N * K) ? __ldg(src + 1)
                                                                                                : make_uint4(0u, 0u, 0u, 0u);
        w[0] = v0.x, w[1] = v0.y, w[2] = v0.z, w[3] = v0.w, w[4] = v1.x, w[5] = v1.y, w[6] = v1.z, w[7] = v1.w;
        s = __ldg(scale_w + n);
    }
    // the row's scale times 1/sqrt(B) as a double-float (sh + sl)
    const float sh = __fmul_rn(s, ch);
    const float sl = __fmaf_rn(s, cl, __fmaf_rn(s, ch, -sh));
    float e[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) codes_to_f32x4(w[k], &e[4 * k]);
    fwht32<LOGB>(e, lane);  // exact: integer sums below 2^15
    uint32_t pk[16];
    // per group of 8 values, the smallest distance (mod 2^16) of a low half
    // above 0x7ffc, kept per 16-bit lane: the low halves of p0 and p1 are
    // packed into one word and 0x7ffc7ffc is subtracted from it as a 32-bit
    // number; a borrow out of the lower lane shifts the upper lane's window by
    // one step, so a lane value <= 8 covers every low half within 2.5 steps
    // of 0x8000 either way
    uint32_t near[4] = {~0u, ~0u, ~0u, ~0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float p0 = e[2 * i], p1 = e[2 * i + 1];
        mul2c(p0, p1, sh);
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        pk[i] = *reinterpret_cast<const uint32_t *>(&h);
        const uint32_t d = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x5410) - 0x7ffc7ffcu;
        asm("min.u16x2 %0, %0, %1;" : "+r"(near[i >> 2]) : "r"(d));
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if ((near[g] & 0xffffu) <= 8u || (near[g] >> 16) <= 8u) {
#pragma unroll
            for (int i = 8 * g; i < 8 * g + 8; ++i) {
                // u * (sh + sl) as hi + lo: the product u * sh exactly, plus u * sl
                const float hi = __fmul_rn(e[i], sh);
                const float lo = __fmaf_rn(e[i], sl, __fmaf_rn(e[i], sh, -hi));
                float rh, rlo;
                fast_two_sum(hi, lo, rh, rlo);
                const uint32_t b = df_to_bf16(rh, rlo);
                pk[i >> 1] = (i & 1) ? ((pk[i >> 1] & 0xffffu) | (b << 16)) : ((pk[i >> 1] & 0xffff0000u) | b);
            }
        }
    }
    const int slot = rl ^ (8 * (c & 7));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        dtile[(32 * c + 2 * i) * kDeqRows + slot] = (uint16_t)(pk[i] & 0xffffu);
        dtile[(32 * c + 2 * i + 1) * kDeqRows + slot] = (uint16_t)(pk[i] >> 16);
    }
    __syncthreads();
    for (int idx = tid; idx < KT * (kDeqRows / 8); idx += blockDim.x) {
        const int kl = idx >> 3, g = idx & 7;
        if (k0 + kl >= K) continue;
        const uint4 v = *reinterpret_cast<const uint4 *>(&dtile[kl * kDeqRows + 8 * (g ^ ((kl >> 5) & 7))]);
        const int64_t nn = n0 + 8 * g;
        uint16_t *dst = T + (k0 + kl) * N + nn;
        if (nn + 8 <= N) {
            if (CR_SPAN((k0 + kl) * N + nn, 8, K * N)) *reinterpret_cast<uint4 *>(dst) = v;
        } else {
            const uint32_t q[4] = {v.x, v.y, v.z, v.w};
            for (int j = 0; j < 8 && nn + j < N; ++j)
                if (CR_SPAN((k0 + kl) * N + nn + j, 1, K * N)) dst[j] = (uint16_t)(q[j >> 1] >> (16 * (j & 1)));
        }
    }
}

}  // namespace

cudaError_t launch_dequant_t(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, uint16_t *T,
                             cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const double c = 1.0 / sqrt((double)block);
    const float ch = (float)c;
    const float cl = (float)(c - (double)ch);
    const int kt = block > 128 ? block : 128;
    dim3 grid((unsigned)((N + kDeqRows - 1) / kDeqRows), (unsigned)((K + kt - 1) / kt));
    const int threads = 2 * kt;  // 64 rows x kt / 32 threads per row
    switch (block) {
        case 8: dequant_t_kernel<8><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
        case 16: dequant_t_kernel<16><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
        case 32: dequant_t_kernel<32><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
        case 64: dequant_t_kernel<64><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
        case 128: dequant_t_kernel<128><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
        default: dequant_t_kernel<256><<<grid, threads, 0, st>>>(Wq, scale_w, N, K, ch, cl, T); break;
    }
    return cudaGetLastError();
}

}  // namespace convrot
