// The int8 backward of a frozen ConvRot layer, second reading.
//
// The pages say only that the input gradient goes through the same fused int8
// GEMM as the forward (MOSS-Image LoRA training guide, sections 4.1 and 7.1;
// sd-scripts PR #2461, Summary).  This reading keeps the weight codes as they
// are stored and moves the weight scale and the rotation around them:
//   D   = fp32(dY[m, n] * s_w[n]),   Dq, s_d = per-row absmax codes of D (no rotation)
//   P   = s_d[m] * sum_n Dq[m, n] Wq[n, k]        (exact int32 sum, then fp32)
//   dX  = bf16( P R )                              (R along K, blocks of b)
// since dY (s_w (.) Wq) R = (dY diag(s_w)) Wq R.  Kernels:
//   scaleq_kernel        D and its codes (fp16-held) and s_d, 32 elements per thread;
//   transpose_widen      Wq [N, K] int8 -> fp16 [K, N] (the GEMM's K-major operand, transient);
//   the GEMM in its fp32-scaled mode writes P (gemm_tc.cu);
//   rot_rows_f32_kernel  the rotation of P's rows and the bf16 rounding.
#include "common.cuh"
#include "fwht.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "wide.cuh"

namespace convrot {
namespace {

constexpr int kThreads = 512;

// Codes of D = dY * colscale per row, without rotation: one row per group of
// G threads, 32 consecutive elements per thread.  A thread keeps the same
// columns for every row, so the block stages its column scales once in shared
// memory, laid out [s][v][t] as float4 so that a warp's read of them is
// contiguous.  The next row's loads are issued before this row's reduction,
// and the partial maxima alternate between two shared arrays so one barrier
// per row suffices.
template <int S>
__global__ void __launch_bounds__(kThreads, S == 1 ? 2 : 1) scaleq_kernel(const uint16_t *x, int64_t rows, int64_t L,
                                                                          const float *colscale, int G, __half *q,
                                                                          float *scale) {
    extern __shared__ float4 cs_s[];  // [S][8][G]
    __shared__ float red[2][kThreads / 32];
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int groups = blockDim.x / G;
    const int wpg = G >> 5;
    const int64_t chunks = L >> 5;
    const int64_t nblocks = (rows + groups - 1) / groups;

    for (int i = threadIdx.x; i < S * 8 * G; i += blockDim.x) {
        const int s = i / (8 * G), v = (i / G) & 7, tt = i % G;
        const int64_t c = (int64_t)s * G + tt;
        cs_s[i] = c < chunks && CR_SPAN(32 * c + 4 * v, 4, L) ? __ldg(reinterpret_cast<const float4 *>(colscale + 32 * c) + v)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    uint32_t raw[S][16];
    auto fetch = [&](int64_t blk) {
        const int64_t row = blk * groups + g;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (c < chunks && row < rows && CR_SPAN(row * L + 32 * c, 32, rows * L)) {
                ld256(x + row * L + 32 * c, raw[s]);
                ld256(x + row * L + 32 * c + 16, raw[s] + 8);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) raw[s][i] = 0u;
            }
        }
    };

    int par = 0;
    int64_t blk = blockIdx.x;
    if (blk < nblocks) fetch(blk);
    for (; blk < nblocks; blk += gridDim.x, par ^= 1) {
        const int64_t row = blk * groups + g;
        float e[S][32];
#pragma unroll
        for (int s = 0; s < S; ++s) unpack_bf16x32(raw[s], e[s]);
        if (blk + gridDim.x < nblocks) fetch(blk + gridDim.x);
        float amax = 0.f;
#pragma unroll
        for (int s = 0; s < S; ++s) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = cs_s[(s * 8 + v) * G + t];
                e[s][4 * v] = __fmul_rn(e[s][4 * v], f.x);
                e[s][4 * v + 1] = __fmul_rn(e[s][4 * v + 1], f.y);
                e[s][4 * v + 2] = __fmul_rn(e[s][4 * v + 2], f.z);
                e[s][4 * v + 3] = __fmul_rn(e[s][4 * v + 3], f.w);
            }
            amax = fmaxf(amax, amax32(e[s]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[par][warp] = amax;
        __syncthreads();
        float m = 0.f;
        for (int w = 0; w < wpg; ++w) m = fmaxf(m, red[par][g * wpg + w]);
        if (row < rows) {
            const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
            if (t == 0 && CR_SPAN(row, 1, rows)) scale[row] = __fdiv_rn(m, 127.f);
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int64_t c = (int64_t)s * G + t;
                if (c < chunks && CR_SPAN(row * L + 32 * c, 32, rows * L)) store_codes32(e[s], inv, q + row * L + 32 * c);
            }
        }
    }
}

// int8 [N, K] -> fp16 [K, N] holding the same integers: a 64 x 64 tile per
// CTA of 256 threads, through a padded shared tile.
__global__ void __launch_bounds__(256) transpose_widen_kernel(const int8_t *W, int64_t N, int64_t K, __half *T) {
    __shared__ int tile[64][65];
    const int t = threadIdx.x;
    const int64_t k0 = (int64_t)blockIdx.x * 64, n0 = (int64_t)blockIdx.y * 64;
    {
        const int r = t >> 2, c = (t & 3) * 16;  // row n0 + r, columns k0 + c .. + 15
        const int64_t n = n0 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < N && k0 + c < K && CR_SPAN(n * K + k0 + c, 16, N * K)) v = __ldg(reinterpret_cast<const uint4 *>(W + n * K + k0 + c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) tile[r][c + i] = (int)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
    }
    __syncthreads();
    const int r = t >> 2, c = (t & 3) * 16;  // output row k0 + r, columns n0 + c .. + 15
    const int64_t k = k0 + r;
    if (k < K && n0 + c < N && CR_SPAN(k * N + n0 + c, 16, K * N)) {
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half2 h = __halves2half2(__int2half_rn(tile[c + 2 * i][r]), __int2half_rn(tile[c + 2 * i + 1][r]));
            o[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(T + k * N + n0 + c);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// dX = bf16(P R): rows of fp32, 32 consecutive elements per thread, the
// Walsh-Hadamard transform in registers and across lanes, times 1/sqrt(b).
template <int LOGB, int S>
__global__ void __launch_bounds__(kThreads) rot_rows_f32_kernel(const float *P, int64_t rows, int64_t L, int G,
                                                                float inv_sqrt_b, uint16_t *out) {
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int groups = blockDim.x / G;
    const int64_t chunks = L >> 5;
    for (int64_t blk = blockIdx.x; blk * groups < rows; blk += gridDim.x) {
        const int64_t row = blk * groups + g;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            float e[32];
            if (c < chunks && row < rows && CR_SPAN(row * L + 32 * c, 32, rows * L)) {
                uint32_t raw[32];
#pragma unroll
                for (int v = 0; v < 4; ++v) ld256(P + row * L + 32 * c + 8 * v, raw + 8 * v);
#pragma unroll
                for (int i = 0; i < 32; ++i) e[i] = __uint_as_float(raw[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) e[i] = 0.f;
            }
            fwht32<LOGB>(e, lane);
            if (c < chunks && row < rows && CR_SPAN(row * L + 32 * c, 32, rows * L)) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(e[2 * i], inv_sqrt_b),
                                                                   __fmul_rn(e[2 * i + 1], inv_sqrt_b));
                    w[i] = *reinterpret_cast<const uint32_t *>(&h);
                }
                uint16_t *dst = out + row * L + 32 * c;
                st256(dst, w);
                st256(dst + 16, w + 8);
            }
        }
    }
}

void shape32(int64_t len, int &G, int &S) {
    const int64_t chunks = len / 32;
    if (chunks <= kThreads) {
        G = (int)((chunks + 31) / 32 * 32);
        S = 1;
    } else {
        G = kThreads;
        S = (int)((chunks + kThreads - 1) / kThreads);
    }
}

int64_t grid_for(int64_t nblocks) {
    const int64_t cap = (int64_t)sm_count() * 2;
    return nblocks < cap ? nblocks : cap;
}

template <int LOGB>
cudaError_t launch_rot_t(const float *P, int64_t rows, int64_t L, int G, int S, float isb, uint16_t *out,
                         cudaStream_t st) {
    const int groups = G >= kThreads ? 1 : kThreads / G;
    const int64_t grid = grid_for((rows + groups - 1) / groups);
    if (S == 1)
        rot_rows_f32_kernel<LOGB, 1><<<(unsigned)grid, groups * G, 0, st>>>(P, rows, L, G, isb, out);
    else
        rot_rows_f32_kernel<LOGB, 2><<<(unsigned)grid, groups * G, 0, st>>>(P, rows, L, G, isb, out);
    return cudaGetLastError();
}

}  // namespace

bool bwd_r2_ok(int64_t N, int64_t K, const void *dY, const void *dX) {
    // rows of 32-element chunks, at most 2 per thread, and 32-byte accesses
    return N % 32 == 0 && K % 32 == 0 && N <= 2 * 32 * kThreads && K <= 2 * 32 * kThreads &&
           ((uintptr_t)dY & 31u) == 0 && ((uintptr_t)dX & 31u) == 0;
}

cudaError_t launch_scaleq(const uint16_t *dY, int64_t M, int64_t N, const float *colscale, uint16_t *q, float *scale,
                          cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    int G, S;
    shape32(N, G, S);
    const int groups = G >= kThreads ? 1 : kThreads / G;
    const int64_t grid = grid_for((M + groups - 1) / groups);
    __half *qh = reinterpret_cast<__half *>(q);
    const int smem = S * 8 * G * (int)sizeof(float4);
    const void *fn = S == 1 ? (const void *)scaleq_kernel<1> : (const void *)scaleq_kernel<2>;
    const cudaError_t e = ensure_smem_attr(fn, smem);
    if (e != cudaSuccess) return e;
    if (S == 1)
        scaleq_kernel<1><<<(unsigned)grid, groups * G, smem, st>>>(dY, M, N, colscale, G, qh, scale);
    else
        scaleq_kernel<2><<<(unsigned)grid, groups * G, smem, st>>>(dY, M, N, colscale, G, qh, scale);
    return cudaGetLastError();
}

cudaError_t launch_transpose_widen(const int8_t *W, int64_t N, int64_t K, uint16_t *T, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    dim3 grid((unsigned)((K + 63) / 64), (unsigned)((N + 63) / 64));
    transpose_widen_kernel<<<grid, 256, 0, st>>>(W, N, K, reinterpret_cast<__half *>(T));
    return cudaGetLastError();
}

cudaError_t launch_rot_rows_f32(const float *P, int64_t rows, int64_t L, int block, uint16_t *out, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    int G, S;
    shape32(L, G, S);
    const float isb = (float)(1.0 / sqrt((double)block));
    switch (block) {
        case 8: return launch_rot_t<3>(P, rows, L, G, S, isb, out, st);
        case 16: return launch_rot_t<4>(P, rows, L, G, S, isb, out, st);
        case 32: return launch_rot_t<5>(P, rows, L, G, S, isb, out, st);
        case 64: return launch_rot_t<6>(P, rows, L, G, S, isb, out, st);
        case 128: return launch_rot_t<7>(P, rows, L, G, S, isb, out, st);
        default: return launch_rot_t<8>(P, rows, L, G, S, isb, out, st);
    }
}

}  // namespace convrot
