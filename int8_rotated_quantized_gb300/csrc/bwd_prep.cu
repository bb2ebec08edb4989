// Backward weights of a frozen ConvRot base, in double-float arithmetic: the
// one-off int8 backward weight, and the transient bf16 weight of the default
// bf16 backward mode (MOSS-Image LoRA training guide, section 4.1: the
// backward option takes bf16 or int8; sd-scripts PR #2461, Summary).
//
// The input gradient goes through the same fused int8 GEMM as the forward
// (MOSS-Image LoRA training guide, sections 4.1 and 7.1, the int8 backward
// option; sd-scripts PR #2461, Summary: frozen base, grad_x only), so its
// weight operand is a ConvRot quantization along the new contraction
// dimension N:
//   W_eff  = (scale_w (.) Wq) R        (the dequantized base, original basis)
//   WtQ    = codes of the rows of W_eff^T rotated along N, scale_wt per row.
//
// Precision.  The rotation of the integer codes along K is exact in fp32
// (|sums| <= 127 * 256).  The scaled values and the rotation along N are kept
// as double-float pairs (hi + lo, two fp32 values, about 48 significant
// bits): products come exact from fused multiply-adds, sums from the
// error-free two-sum.  The code decision is then taken in fp32 on the
// fp32-rounded transform (the hi part), as everywhere else.  This replaces fp64
// arithmetic, which this GPU executes at a small fraction of its fp32 rate.
//
// Kernel 1 (prep_transpose_df_kernel): a CTA takes 16 weight rows and one
// Hadamard block of b columns, transforms each row segment, scales it and
// writes the transposed tile T[k][n] as (hi, lo) pairs.
// Kernel 2 (rotq_df_kernel): each row of T (length N) is transformed along N
// in blocks of b and quantized per row, 8 elements per thread, blocks wider
// than 8 spread over b/8 consecutive lanes.
#include "common.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "wide.cuh"

namespace convrot {
namespace {

// ------------------------------------------------------------ double-float --

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

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

constexpr int kPrepRows = 16;
constexpr int kThreads = 512;

// T[k][n] = (scale_w[n] * (H_b q_n)[k]) / sqrt(b) as (hi, lo).
__global__ void __launch_bounds__(256) prep_transpose_df_kernel(const int8_t *Wq, const float *scale_w, int64_t N,
                                                                int64_t K, int b, float ch, float cl, float2 *T) {
    // [b][kPrepRows]; the row slot is xor-swizzled with the 8-column group so
    // that the 16 lanes writing one row land in 16 distinct bank pairs.
    extern __shared__ float2 tile[];
    const int lanes = b >> 3;
    const int64_t n0 = (int64_t)blockIdx.x * kPrepRows;
    const int64_t k0 = (int64_t)blockIdx.y * b;
    const int total = kPrepRows * lanes;
    const int lane = threadIdx.x & 31;
    for (int j0 = 0; j0 < total; j0 += blockDim.x) {
        if (j0 + (int)(threadIdx.x & ~31u) >= total) break;  // warp-uniform
        const int j = j0 + threadIdx.x;
        const bool valid = j < total;
        const int rl = valid ? j / lanes : 0;
        const int cb = valid ? j - rl * lanes : 0;
        const int64_t n = n0 + rl;
        float e[8];
        if (valid && n < N) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(Wq + n * K + k0 + 8 * cb));
            const uint32_t w[2] = {v.x, v.y};
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = (float)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = 0.f;
        }
        // exact integer transform along K (in-thread stages, then across lanes)
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((i & h) == 0) {
                    const float a = e[i], c = e[i + h];
                    e[i] = a + c;
                    e[i + h] = a - c;
                }
        for (int m = 1; m < lanes; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float p = __shfl_xor_sync(0xffffffffu, e[i], m);
                e[i] = upper ? (p - e[i]) : (e[i] + p);
            }
        }
        const float s = (valid && n < N) ? __ldg(scale_w + n) : 0.f;
        if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // s * u is exact as a pair (24 + 15 significant bits); then * (1/sqrt(b)).
                const float p = __fmul_rn(s, e[i]);
                const float pe = __fmaf_rn(s, e[i], -p);
                float rh, rlo;
                df_mul(p, pe, ch, cl, rh, rlo);
                tile[(8 * cb + i) * kPrepRows + (rl ^ (cb & (kPrepRows - 1)))] = make_float2(rh, rlo);
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < b * kPrepRows; idx += blockDim.x) {
        const int kl = idx / kPrepRows;
        const int rl = idx - kl * kPrepRows;
        if (n0 + rl < N) T[(k0 + kl) * N + n0 + rl] = tile[kl * kPrepRows + (rl ^ ((kl >> 3) & (kPrepRows - 1)))];
    }
}

// Rotate + quantize rows of double-float values (length L) along the row.
template <int S>
__global__ void __launch_bounds__(kThreads) rotq_df_kernel(const float2 *T, int64_t rows, int64_t L, int lanes,
                                                          float scale_denom, int8_t *q, float *scale) {
    __shared__ float red[kThreads / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int G = blockDim.x;
    const int t = threadIdx.x;
    const int64_t chunks = L >> 3;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        float eh[S][8], el[S][8];
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (c < chunks) {
                const float4 *p = reinterpret_cast<const float4 *>(T + row * L + 8 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = __ldcs(p + i);
                    eh[s][2 * i] = v.x, el[s][2 * i] = v.y, eh[s][2 * i + 1] = v.z, el[s][2 * i + 1] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) eh[s][i] = el[s][i] = 0.f;
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int s = 0; s < S; ++s) {
#pragma unroll
            for (int h = 1; h < 8; h <<= 1)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if ((i & h) == 0) {
                        float sh, sl, dh, dl;
                        df_add(eh[s][i], el[s][i], eh[s][i + h], el[s][i + h], sh, sl);
                        df_add(eh[s][i], el[s][i], -eh[s][i + h], -el[s][i + h], dh, dl);
                        eh[s][i] = sh, el[s][i] = sl, eh[s][i + h] = dh, el[s][i + h] = dl;
                    }
            for (int m = 1; m < lanes; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float ph = __shfl_xor_sync(0xffffffffu, eh[s][i], m);
                    const float pl = __shfl_xor_sync(0xffffffffu, el[s][i], m);
                    float rh, rl;
                    if (upper)
                        df_add(ph, pl, -eh[s][i], -el[s][i], rh, rl);
                    else
                        df_add(eh[s][i], el[s][i], ph, pl, rh, rl);
                    eh[s][i] = rh, el[s][i] = rl;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(eh[s][i]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        float m = 0.f;
        for (int w = 0; w < (G >> 5); ++w) m = fmaxf(m, red[w]);
        __syncthreads();  // red is rewritten by the next row
        // fp32 decision on the fp32-rounded transform (hi), as everywhere else.
        const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
        if (t == 0) scale[row] = __fdiv_rn(m, scale_denom);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (c >= chunks) continue;
            uint32_t w[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int qi = max(-127, min(127, __float2int_rn(__fmul_rn(eh[s][i], inv))));
                w[i >> 2] |= (uint32_t)(qi & 0xff) << (8 * (i & 3));
            }
            *reinterpret_cast<uint2 *>(q + row * L + 8 * c) = make_uint2(w[0], w[1]);
        }
    }
}

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
    if (ok) {
        const uint4 *src = reinterpret_cast<const uint4 *>(Wq + n * K + k0 + 32 * c);
        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
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
            *reinterpret_cast<uint4 *>(dst) = v;
        } else {
            const uint32_t q[4] = {v.x, v.y, v.z, v.w};
            for (int j = 0; j < 8 && nn + j < N; ++j) dst[j] = (uint16_t)(q[j >> 1] >> (16 * (j & 1)));
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

cudaError_t launch_bwd_prep_df(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, void *work,
                               int8_t *WtQ, float *scale_wt, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    float2 *T = static_cast<float2 *>(work);
    // 1/sqrt(b) as a double-float constant
    const double c = 1.0 / sqrt((double)block);
    const float ch = (float)c;
    const float cl = (float)(c - (double)ch);
    const size_t smem = sizeof(float2) * (size_t)block * kPrepRows;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(prep_transpose_df_kernel),
                                     (int)(sizeof(float2) * 256 * kPrepRows));
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((N + kPrepRows - 1) / kPrepRows), (unsigned)(K / block));
    prep_transpose_df_kernel<<<grid, 256, smem, st>>>(Wq, scale_w, N, K, block, ch, cl, T);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // rows of T: length N, 8 elements per thread, 512 threads, S slots
    const int64_t chunks = N / 8;
    const int S = chunks <= kThreads ? 1 : chunks <= 2 * kThreads ? 2 : chunks <= 4 * kThreads ? 4 : 8;
    const int sms = sm_count();
    const int64_t g = K < (int64_t)sms * 2 ? K : (int64_t)sms * 2;
    const float denom = (float)(127.0 * sqrt((double)block));
    const int lanes = block / 8;
    switch (S) {
        case 1: rotq_df_kernel<1><<<(unsigned)g, kThreads, 0, st>>>(T, K, N, lanes, denom, WtQ, scale_wt); break;
        case 2: rotq_df_kernel<2><<<(unsigned)g, kThreads, 0, st>>>(T, K, N, lanes, denom, WtQ, scale_wt); break;
        case 4: rotq_df_kernel<4><<<(unsigned)g, kThreads, 0, st>>>(T, K, N, lanes, denom, WtQ, scale_wt); break;
        default: rotq_df_kernel<8><<<(unsigned)g, kThreads, 0, st>>>(T, K, N, lanes, denom, WtQ, scale_wt); break;
    }
    return cudaGetLastError();
}

}  // namespace convrot
