// The one-off int8 backward weight of a frozen ConvRot base.
//
// The input gradient goes through the same fused int8 GEMM as the forward
// (MOSS-Image LoRA training guide, sections 4.1 and 7.1, the int8 backward
// option; sd-scripts PR #2461, Summary: frozen base, grad_x only), so its
// weight operand is a ConvRot quantization along the new contraction
// dimension N:
//   W_eff  = (scale_w (.) Wq) R        (the dequantized base, original basis)
//   WtQ    = codes of the rows of W_eff^T rotated along N, scale_wt per row.
// With E = the integer transform of the codes along K (exact) and
// p[n, k] = scale_w[n] E[n, k] / sqrt(b), row k of the result is
//   u[k, n'] = sum over n in the block of n' of H[n', n] p[n, k],
//   scale_wt[k] = m_k / (127 sqrt(b)) and codes rne(u * (127 / m_k)), m_k = max |u[k, :]|,
// where every u is the fp32 rounding of the exact value (the code decision is
// taken in fp32 on it, as everywhere else).
//
// Two kernels, neither of which keeps W_eff in memory:
//   1. approximate pass (tile of T = max(128, b) weight rows x T columns): the
//      exact integer transform along K, a transposed int16 copy of E in shared
//      memory, p and its transform along N in plain fp32, and per tile column
//      the largest |u| with a bound delta on its error,
//        delta = (4 + log2 b) 2^-24 sqrt(b) ||p||_2 >= (4 + log2 b) 2^-24 sum |p|
//        over any block (products, 1/sqrt(b) and the log2 b butterfly stages
//        each round once per value; the error of any value is at most its share
//        of 2^-24 times the magnitudes summed; Cauchy-Schwarz for the norm);
//      Each tile column raises the column's running lower bound lb[k] to
//      max - delta (atomic max) and reads it back: if max + delta still
//      reaches it, the values within 2 delta of the tile's maximum (usually
//      one) are recomputed exactly in double-float arithmetic (about 48
//      significant bits) and the largest raises m[k] (atomic max).  The tile
//      holding the column's maximum always does (its upper bound is at least
//      every lower bound), so m[k] ends exact; in a random order of tiles only
//      about ln(n)/n of the n tiles of a column set a new bound;
//   2. codes pass: the same approximate transform; a code whose scaled value
//      lies farther than the error margin from a rounding boundary (k + 1/2)
//      is the code of the exact value; the few others (about 3 in 10^4) are
//      recomputed exactly in double-float by the warp that holds them.
// The caller's workspace holds lb and m (2 K floats, cleared by the launcher).
//
// Shared-memory layout of the int16 E^T tile [T][T]: the 16-byte group g of
// row k is stored at group g ^ swz(k), which makes both the transposing
// stores of the first phase (32 lanes writing one row each of 4 or 8
// columns) and the 16-byte loads of the second phase (8 lanes reading 2 or 1
// columns) free of bank conflicts.
#include "common.cuh"
#include "dfloat.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "wide.cuh"

namespace convrot {
namespace {

constexpr int kWtThreads = 512;

template <int LOGB>
struct WtShape {
    static constexpr int B = 1 << LOGB;
    static constexpr int T = B > 128 ? B : 128;       // weight rows n and columns k of a tile
    static constexpr int LPR = T / 32;                // lanes per tile row (phase 1) / column (phase 2)
    static constexpr int PER = T * LPR / kWtThreads;  // 32-element items per thread per phase
    static constexpr int ET_BYTES = T * T * 2;
    // Staging the next tile's codes in shared memory (cp.async, two buffers) while
    // the current one is processed measured slower on GB300 (0.22 ms against
    // 0.20 ms for 16384 x 4096: the larger footprint costs occupancy), so each CTA
    // takes one tile and loads its codes directly.
    static constexpr bool PF = false;
    // E^T, codes, row scales (two buffers with PF) and, with PF, two buffers of codes [T][T + 16]
    static constexpr int SMEM = ET_BYTES + T * T + (PF ? 2 : 1) * T * 4 + (PF ? 2 * T * (T + 16) : 0);
    // (4 + log2 b) 2^-24 sqrt(b), with slack for the rounding of the norm itself
    static constexpr float kDelta = (4.0f + LOGB) * 5.9604645e-08f * (LOGB == 3   ? 2.8284271f
                                                                      : LOGB == 4 ? 4.0f
                                                                      : LOGB == 5 ? 5.6568542f
                                                                      : LOGB == 6 ? 8.0f
                                                                      : LOGB == 7 ? 11.313708f
                                                                                  : 16.0f) * 1.01f;
};

template <int LPR>
__device__ __forceinline__ int et_swz(int k) {
    return LPR == 4 ? (((k >> 5) & 3) | ((k & 1) << 2)) : ((k >> 5) & 7);
}

// (q0, q1) <- (a0 * a0 + q0, a1 * a1 + q1), one rounding per lane.
__device__ __forceinline__ void sq2acc(float &q0, float &q1, float a0, float a1) {
    asm("{\n .reg .b64 rq, ra;\n mov.b64 rq, {%0, %1};\n mov.b64 ra, {%2, %3};\n"
        " fma.rn.f32x2 rq, ra, ra, rq;\n mov.b64 {%0, %1}, rq;\n}"
        : "+f"(q0), "+f"(q1)
        : "f"(a0), "f"(a1));
}

// Transform along N of a column item held as e[8q + r] <-> tile row
// n = 8 LPR q + 8 c + r (c = lane % LPR): fp32 butterflies (packed pairs
// where the partners sit in different register pairs), stages h < B.
template <int LOGB, int LPR>
__device__ __forceinline__ void fwht_cols(float (&e)[32], int lane) {
    constexpr int B = 1 << LOGB;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float a = e[i], c = e[i + 1];
        e[i] = a + c;
        e[i + 1] = a - c;
    }
#pragma unroll
    for (int h = 2; h < 8 && h < B; h <<= 1)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            if ((i & h) == 0) addsub2(e[i], e[i + 1], e[i + h], e[i + h + 1]);
#pragma unroll
    for (int m = 1; m < LPR && 8 * m < B; m <<= 1) {
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
#pragma unroll
    for (int hq = 8; hq < 32 && 8 * LPR * (hq / 8) < B; hq <<= 1)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            if ((i & hq) == 0) addsub2(e[i], e[i + 1], e[i + hq], e[i + hq + 1]);
}

// int16 pair word -> two fp32 values of the same integers (bias by 2^15, splice
// under the exponent of 2^23, subtract 2^23 + 2^15 exactly).
__device__ __forceinline__ void i16x2_to_f32(uint32_t w, float &lo, float &hi) {
    const uint32_t x = w ^ 0x80008000u;
    lo = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7610));
    hi = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7632));
    add2c(lo, hi, -8421376.0f);
}

// Exact u for tile column kk and tile row np (both of this CTA), rounded to
// fp32: the warp sums, in double-float, s_n E[n, kk] with the signs of H over
// the b rows of np's block, then multiplies by (ch + cl) = 1/sqrt(b).  Every
// lane returns the same value (the double-float sum is commutative).
template <int LOGB, int LPR>
__device__ __forceinline__ float exact_u(const uint8_t *et, const float *ss, int kk, int np, float ch, float cl,
                                         int lane) {
    constexpr int B = 1 << LOGB;
    constexpr int T = 32 * LPR;
    const int blk0 = np & ~(B - 1), rel = np - blk0;
    float hi = 0.f, lo = 0.f;
    const uint8_t *row = et + kk * (2 * T);
    for (int idx = lane; idx < B; idx += 32) {
        const int n = blk0 + idx;
        const int16_t E = *reinterpret_cast<const int16_t *>(row + (((n >> 3) ^ et_swz<LPR>(kk)) << 4) + ((n & 7) << 1));
        const float s = ss[n], ef = (float)E;
        float ph = __fmul_rn(s, ef), pl = __fmaf_rn(s, ef, -ph);
        if (__popc(idx & rel) & 1) ph = -ph, pl = -pl;
        df_add(hi, lo, ph, pl, hi, lo);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, m), ol = __shfl_xor_sync(0xffffffffu, lo, m);
        df_add(hi, lo, oh, ol, hi, lo);
    }
    float rh, rl;
    df_mul(hi, lo, ch, cl, rh, rl);
    return rh;
}

// PASS 1: the exact column maxima m [K] (float bits, atomic max; lb [K] the
// running lower bounds).  PASS 3: the codes of the tile, into WtQ [K][N], and
// (tiles of the first row) scale_wt [K].  A CTA takes tiles in turn, row
// tiles fastest (with the launch grid of one CTA per tile, one each); with
// S::PF the next tile's codes and row scales are copied into shared memory
// (cp.async, two buffers) while the current one is processed.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes) : "memory");
}

template <int LOGB, int PASS>
__global__ void __launch_bounds__(kWtThreads, WtShape<LOGB>::T == 128 ? 2 : 1) wtq_tile_kernel(const int8_t *Wq, const float *scale_w, int64_t N,
                                                              int64_t K, float ch, float cl, unsigned *lb, unsigned *m,
                                                              float scale_denom, float *scale_wt, int8_t *WtQ) {
    using S = WtShape<LOGB>;
    constexpr int T = S::T, LPR = S::LPR;
    constexpr bool PF = S::PF;
    constexpr int QROW = T + 16;  // padded rows of the staged codes: conflict-free 16-byte reads
    extern __shared__ __align__(16) uint8_t wsm[];
    uint8_t *et = wsm;
    int8_t *ct = reinterpret_cast<int8_t *>(wsm + S::ET_BYTES);
    float *ssb = reinterpret_cast<float *>(wsm + S::ET_BYTES + T * T);  // [PF ? 2 : 1][T]
    uint8_t *qs = wsm + S::ET_BYTES + T * T + (PF ? 2 : 1) * T * 4;     // [2][T][QROW] when PF
    const int lane = threadIdx.x & 31;
    const int64_t ntn = (N + T - 1) / T, ntk = (K + T - 1) / T, tiles = ntn * ntk;

    auto prefetch = [&](int64_t tile, int buf) {
        const int64_t pn0 = (tile % ntn) * T, pk0 = (tile / ntn) * T;
        for (int q = threadIdx.x; q < T * (T / 16); q += kWtThreads) {
            const int r = q / (T / 16), j = q - r * (T / 16);
            const int64_t n = pn0 + r, k = pk0 + 16 * j;
            const bool ok = n < N && k < K;
            cp_async16(qs + (buf * T + r) * QROW + 16 * j, ok ? Wq + n * K + k : Wq, ok ? 16 : 0);
        }
        for (int q = threadIdx.x; q < T / 4; q += kWtThreads) {  // N is a multiple of 16: whole groups of 4
            const int64_t n = pn0 + 4 * q;
            cp_async16(ssb + buf * T + 4 * q, n < N ? scale_w + n : scale_w, n < N ? 16 : 0);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    int buf = 0;
    if constexpr (PF) {
        if ((int64_t)blockIdx.x < tiles) prefetch(blockIdx.x, 0);
    }
#pragma unroll 1
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, buf ^= PF ? 1 : 0) {
    const int tn = (int)(tile % ntn);
    const int64_t n0 = (int64_t)tn * T, k0 = (tile / ntn) * T;
    float *ss = ssb + buf * T;
    if constexpr (PF) {
        if (tile + gridDim.x < tiles) {
            prefetch(tile + gridDim.x, buf ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // this tile's codes and scales are in buffer buf for every thread
    }

    // phase 1: exact transform along K of the tile's rows, stored transposed as int16
#pragma unroll 1
    for (int it = 0; it < S::PER; ++it) {
        const int item = threadIdx.x + it * kWtThreads;
        const int r = item / LPR, c = item - r * LPR;
        const int64_t n = n0 + r, k = k0 + 32 * c;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if constexpr (PF) {  // staged (zeros outside the matrix)
            const uint4 *src = reinterpret_cast<const uint4 *>(qs + (buf * T + r) * QROW + 32 * c);
            const uint4 v0 = src[0], v1 = src[1];
            w[0] = v0.x, w[1] = v0.y, w[2] = v0.z, w[3] = v0.w, w[4] = v1.x, w[5] = v1.y, w[6] = v1.z, w[7] = v1.w;
        } else if (n < N && k < K && CR_SPAN(n * K + k, 16, N * K)) {  // K is a multiple of 16: the second 16 codes may lie past the row
            const uint4 *src = reinterpret_cast<const uint4 *>(Wq + n * K + k);
            const uint4 v0 = __ldg(src);
            const uint4 v1 = k + 16 < K && CR_SPAN(n * K + k + 16, 16, N * K) ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
            w[0] = v0.x, w[1] = v0.y, w[2] = v0.z, w[3] = v0.w, w[4] = v1.x, w[5] = v1.y, w[6] = v1.z, w[7] = v1.w;
        }
        float e[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) codes_to_f32x4(w[j], &e[4 * j]);
        fwht32<LOGB>(e, lane);  // exact: |sums| <= 127 b < 2^15
        // + 1.5 2^23: the low 16 bits of the sum are the integer as int16
#pragma unroll
        for (int i = 0; i < 32; i += 2) add2c(e[i], e[i + 1], kMagicI8);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int kk = 32 * c + i;
            *reinterpret_cast<uint16_t *>(et + kk * (2 * T) + (((r >> 3) ^ et_swz<LPR>(kk)) << 4) + ((r & 7) << 1)) =
                (uint16_t)(__float_as_uint(e[i]) & 0xffffu);
        }
        if (!PF && c == 0) ss[r] = n < N && CR_SPAN(n, 1, N) ? __ldg(scale_w + n) : 0.f;
    }
    __syncthreads();

    // phase 2: the transform along N of each tile column, approximately in fp32
#pragma unroll 1
    for (int it = 0; it < S::PER; ++it) {
        const int item = threadIdx.x + it * kWtThreads;
        const int kk = item / LPR, c = item - kk * LPR;
        float p[32], q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int g = c + LPR * q;  // rows 8g .. 8g + 7
            const uint4 v = *reinterpret_cast<const uint4 *>(et + kk * (2 * T) + ((g ^ et_swz<LPR>(kk)) << 4));
            i16x2_to_f32(v.x, p[8 * q + 0], p[8 * q + 1]);
            i16x2_to_f32(v.y, p[8 * q + 2], p[8 * q + 3]);
            i16x2_to_f32(v.z, p[8 * q + 4], p[8 * q + 5]);
            i16x2_to_f32(v.w, p[8 * q + 6], p[8 * q + 7]);
            const float4 s0 = *reinterpret_cast<const float4 *>(ss + 8 * g);
            const float4 s1 = *reinterpret_cast<const float4 *>(ss + 8 * g + 4);
            mul2v(p[8 * q + 0], p[8 * q + 1], s0.x, s0.y);
            mul2v(p[8 * q + 2], p[8 * q + 3], s0.z, s0.w);
            mul2v(p[8 * q + 4], p[8 * q + 5], s1.x, s1.y);
            mul2v(p[8 * q + 6], p[8 * q + 7], s1.z, s1.w);
#pragma unroll
            for (int r = 0; r < 8; r += 2) {
                mul2c(p[8 * q + r], p[8 * q + r + 1], ch);
                sq2acc(q0, q1, p[8 * q + r], p[8 * q + r + 1]);
            }
        }
        fwht_cols<LOGB, LPR>(p, lane);
        float ssq = q0 + q1;
#pragma unroll
        for (int s2 = 1; s2 < LPR; s2 <<= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, s2);
        const float delta = sqrtf(ssq) * S::kDelta;
        const int64_t k = k0 + kk;
        if constexpr (PASS == 1) {
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(p[i]));
#pragma unroll
            for (int s2 = 1; s2 < LPR; s2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s2));
            // raise the column's lower bound; does this tile's upper bound still reach it?
            bool need = false;
            if (c == 0 && k < K && CR_SPAN(k, 1, K)) {
                const float mine = fmaxf(mx - delta, 0.f);
                const float cur = fmaxf(__uint_as_float(atomicMax(lb + k, __float_as_uint(mine))), mine);
                need = mx + delta >= cur && mx + delta > 0.f;
            }
            need = __shfl_sync(0xffffffffu, need, lane & ~(LPR - 1)) != 0;
            uint32_t cand = 0u;
            if (need) {
                const float floor_v = mx - 2.f * delta;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (fabsf(p[i]) >= floor_v) cand |= 1u << i;
            }
            float ex = 0.f;  // exact |u| of this lane's candidates
            for (;;) {
                const uint32_t who = __ballot_sync(0xffffffffu, cand != 0u);
                if (who == 0u) break;
                const int src = __ffs(who) - 1;
                const int i = __ffs(__shfl_sync(0xffffffffu, cand, src)) - 1;
                const int kk_s = __shfl_sync(0xffffffffu, kk, src), c_s = __shfl_sync(0xffffffffu, c, src);
                const float u = exact_u<LOGB, LPR>(et, ss, kk_s, 8 * LPR * (i >> 3) + 8 * c_s + (i & 7), ch, cl, lane);
                if (lane == src) {
                    ex = fmaxf(ex, fabsf(u));
                    cand &= ~(1u << i);
                }
            }
#pragma unroll
            for (int s2 = 1; s2 < LPR; s2 <<= 1) ex = fmaxf(ex, __shfl_xor_sync(0xffffffffu, ex, s2));
            if (need && c == 0 && CR_SPAN(k, 1, K)) atomicMax(m + k, __float_as_uint(ex));
        } else {
            const float mk = k < K && CR_SPAN(k, 1, K) ? __uint_as_float(__ldcg(m + k)) : 0.f;
            const float iv = mk > 0.f ? __fdiv_rn(127.f, mk) : 0.f;
            if (tn == 0 && c == 0 && k < K && CR_SPAN(k, 1, K)) scale_wt[k] = __fdiv_rn(mk, scale_denom);
            // |t - t_exact| <= delta * iv + 2^-22 (|u| iv <= 127 + delta iv) + 2^-16 (the fp32 roundings of t)
            const float margin = __fmaf_rn(delta, iv * 1.0000002f, 3.0517578125e-05f + 1.52587890625e-05f);
            const float thr = 0.5f - margin;  // a residual |t - rne(t)| >= thr is near a rounding boundary
            uint32_t flags = 0u;
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float t0 = p[i], t1 = p[i + 1];
                mul2c(t0, t1, iv);
                float m0 = t0, m1 = t1;
                add2c(m0, m1, kMagicI8);  // rne(t) in the low byte (|t| <= 127 + a bound far below 0.5)
                float r0 = m0, r1 = m1;
                add2c(r0, r1, -kMagicI8);
                if (fabsf(t0 - r0) >= thr) flags |= 1u << i;
                if (fabsf(t1 - r1) >= thr) flags |= 2u << i;
                p[i] = m0, p[i + 1] = m1;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = __byte_perm(__float_as_uint(p[4 * j]), __float_as_uint(p[4 * j + 1]), 0x0040);
                const uint32_t hi = __byte_perm(__float_as_uint(p[4 * j + 2]), __float_as_uint(p[4 * j + 3]), 0x0040);
                packed[j] = __byte_perm(lo, hi, 0x5410);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint2 *>(ct + kk * T + 8 * (c + LPR * q)) = make_uint2(packed[2 * q], packed[2 * q + 1]);
            // codes near a rounding boundary: the warp recomputes them exactly, one at a time
            for (;;) {
                const uint32_t who = __ballot_sync(0xffffffffu, flags != 0u);
                if (who == 0u) break;
                const int src = __ffs(who) - 1;
                const int i = __ffs(__shfl_sync(0xffffffffu, flags, src)) - 1;
                const int kk_s = __shfl_sync(0xffffffffu, kk, src), c_s = __shfl_sync(0xffffffffu, c, src);
                const float iv_s = __shfl_sync(0xffffffffu, iv, src);
                const int np = 8 * LPR * (i >> 3) + 8 * c_s + (i & 7);
                const float u = exact_u<LOGB, LPR>(et, ss, kk_s, np, ch, cl, lane);
                if (lane == src) {
                    ct[kk * T + np] = (int8_t)max(-127, min(127, __float2int_rn(__fmul_rn(u, iv))));
                    flags &= ~(1u << i);
                }
            }
        }
    }
    if constexpr (PASS == 3) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < T * (T / 16); idx += kWtThreads) {
            const int kk = idx / (T / 16), g = idx - kk * (T / 16);
            const int64_t k = k0 + kk, n = n0 + 16 * g;
            if (k < K && n < N && CR_SPAN(k * N + n, 16, K * N))
                *reinterpret_cast<uint4 *>(WtQ + k * N + n) = *reinterpret_cast<const uint4 *>(ct + kk * T + 16 * g);
        }
    }
    __syncthreads();  // E^T, the codes tile and this buffer are free for the next tile
    }
}

template <int LOGB>
cudaError_t launch_wtq(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, float ch, float cl, float denom,
                       unsigned *work, int8_t *WtQ, float *scale_wt, cudaStream_t st) {
    using S = WtShape<LOGB>;
    unsigned *lb = work, *m = work + K;
    cudaError_t e = cudaMemsetAsync(work, 0, (size_t)2 * K * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(reinterpret_cast<const void *>(wtq_tile_kernel<LOGB, 1>), S::SMEM);
    if (e == cudaSuccess) e = ensure_smem_attr(reinterpret_cast<const void *>(wtq_tile_kernel<LOGB, 3>), S::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((N + S::T - 1) / S::T) * ((K + S::T - 1) / S::T);
    auto grid_of = [&](const void *kernel) {  // one CTA per tile, unless tiles are staged ahead
        const int64_t resident = (int64_t)sm_count() * blocks_per_sm(kernel, kWtThreads, S::SMEM);
        return (unsigned)(!S::PF || tiles < resident ? tiles : resident);
    };
    auto k1 = wtq_tile_kernel<LOGB, 1>;
    auto k3 = wtq_tile_kernel<LOGB, 3>;
    k1<<<grid_of(reinterpret_cast<const void *>(k1)), kWtThreads, S::SMEM, st>>>(Wq, scale_w, N, K, ch, cl, lb, m,
                                                                                 denom, nullptr, nullptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k3<<<grid_of(reinterpret_cast<const void *>(k3)), kWtThreads, S::SMEM, st>>>(Wq, scale_w, N, K, ch, cl, lb, m,
                                                                                 denom, scale_wt, WtQ);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_weight_work_bytes(int64_t N, int64_t K) {
    (void)N;
    return (size_t)2 * K * sizeof(unsigned);  // per column the running lower bound and the exact maximum
}

cudaError_t launch_bwd_prep_df(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, void *work,
                               int8_t *WtQ, float *scale_wt, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const double c = 1.0 / sqrt((double)block);
    const float ch = (float)c;
    const float cl = (float)(c - (double)ch);
    const float denom = (float)(127.0 * sqrt((double)block));
    unsigned *w = static_cast<unsigned *>(work);
    switch (block) {
        case 8: return launch_wtq<3>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
        case 16: return launch_wtq<4>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
        case 32: return launch_wtq<5>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
        case 64: return launch_wtq<6>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
        case 128: return launch_wtq<7>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
        default: return launch_wtq<8>(Wq, scale_w, N, K, ch, cl, denom, w, WtQ, scale_wt, st);
    }
}

}  // namespace convrot
