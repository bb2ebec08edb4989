// Row-wise kernels of libconvrot with 8 elements per thread: rotate +
// quantize (the LoRA-merging weight quantizer, and rows that the 32-element
// kernels of rotq_wide.cu cannot take: lengths that are not a multiple of 32
// or pointers that are only 16-byte aligned) and the quantized embedding
// lookup for such tables.  The launchers here dispatch to rotq_wide.cu when
// its conditions hold.
//
// The rotation is the block-diagonal normalised Sylvester-Hadamard matrix
// R = I (x) H_b / sqrt(b) (MOSS-Image LoRA training guide, section 7.1,
// ConvRot INT8: the rotation spreads activation outliers over each block
// before quantization).  It is applied as a fast Walsh-Hadamard transform: every thread
// holds 8 consecutive elements of a row (one 16-byte load of bf16), does the
// three in-register butterfly stages, and the remaining log2(b/8) stages run
// across the b/8 consecutive lanes of a warp with __shfl_xor_sync.  The
// butterfly (a, c) -> (a + c, a - c) on indices k and k ^ h reproduces the
// Sylvester ordering H[i][j] = (-1)^popcount(i & j).
//
// Quantization is symmetric and per row (sd-scripts PR #2461, ConvRot INT8,
// Summary: weights and, at run time, activations get one absmax scale per row):
// with u = H_b x the unnormalised transform, amax_u = max |u| over the row,
//   scale = amax_u / (127 sqrt(b))   (= max |x R| / 127),
//   code  = clamp(rne(u * (127 / amax_u)), -127, 127)   (= rne(v / scale)).
// An all-zero row gets scale 0 and codes 0.
#include "common.cuh"
#include "fwht.cuh"
#include "internal.h"
#include "launch_cache.h"

namespace convrot {
namespace {

constexpr int kMaxThreads = 512;

__device__ __forceinline__ float absv(float v) { return fabsf(v); }
__device__ __forceinline__ float maxv(float a, float b) { return fmaxf(a, b); }

// ------------------------------------------------------------------- FWHT --

// In-register stages h = 1, 2, 4 on the 8 elements of one lane.
__device__ __forceinline__ void fwht8(float (&e)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {  // h = 1 lies inside a pair: scalar
        const float a = e[i], c = e[i + 1];
        e[i] = a + c;
        e[i + 1] = a - c;
    }
    addsub2(e[0], e[1], e[2], e[3]);  // h = 2
    addsub2(e[4], e[5], e[6], e[7]);
    addsub2(e[0], e[1], e[4], e[5]);  // h = 4
    addsub2(e[2], e[3], e[6], e[7]);
}

// Cross-lane stages h = 8, 16, ..., b/2 (lane xor masks 1 .. lanes/2).  Every
// lane of the warp must call this with the same `lanes`.
__device__ __forceinline__ void fwht_lanes(float (&e)[8], int lanes, int lane) {
    for (int m = 1; m < lanes; m <<= 1) {
        const float sg = (lane & m) ? -1.f : 1.f;
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(0xffffffffu, e[i], m);
#pragma unroll
        for (int i = 0; i < 8; i += 2) sfma2(sg, e[i], e[i + 1], p[i], p[i + 1]);
    }
}

// ----------------------------------------------------------- code stores --
//
__device__ __forceinline__ void quant_store(float (&e)[8], float inv, int8_t *dst) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) mul2c(e[i], e[i + 1], inv);
#pragma unroll
    for (int i = 0; i < 8; i += 2) add2c(e[i], e[i + 1], kMagicI8);
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = __float_as_uint(e[i]);
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t lo = __byte_perm(b[4 * k], b[4 * k + 1], 0x0040);
        const uint32_t hi = __byte_perm(b[4 * k + 2], b[4 * k + 3], 0x0040);
        w[k] = __byte_perm(lo, hi, 0x5410);
    }
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void quant_store(float (&e)[8], float inv, __half *dst) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) mul2c(e[i], e[i + 1], inv);
#pragma unroll
    for (int i = 0; i < 8; i += 2) add2c(e[i], e[i + 1], kMagicF16);
    const __half2 k1152 = __half2half2(__ushort_as_half((unsigned short)0x6480));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v = __byte_perm(__float_as_uint(e[2 * i]), __float_as_uint(e[2 * i + 1]), 0x5410);
        __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&v), k1152);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// fp16-held codes of 8 integers (the widening of int8 codes).
__device__ __forceinline__ void store_codes(__half *dst, const int (&q)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __halves2half2(__int2half_rn(q[2 * i]), __int2half_rn(q[2 * i + 1]));
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------ rotate + quantize --

struct RotqArgs {
    const void *x;
    int64_t rows, K, ldx;
    int lanes;          // b / 8
    int G;              // threads per row group (multiple of 32, <= 512)
    float scale_denom;  // fp32(127 sqrt(b))
    void *q;            // codes, row stride K
    float *scale;
    const float *lora_A;  // [rank, K]
    const float *lora_B;  // [rows, rank]
    int rank;
    float coef;  // scale * alpha / rank
};

// Raw storage of one 8-element slot of bf16 as loaded (one 16-byte vector), so
// the next rows can be prefetched into registers while the current ones are
// transformed.
struct Raw8 {
    uint4 v;
    __device__ __forceinline__ void load(const uint16_t *p) { v = __ldcs(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ void zero() { v = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void unpack(float (&e)[8]) const {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e[2 * i] = __uint_as_float(w[i] << 16);
            e[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
// x is bf16 (uint16_t bits), the transform fp32.  OutT: int8_t codes or
// __half-held codes.  S: 8-element
// slots per thread.  RPT: rows held per thread group at once.  LORA: merge
// W + coef * B@A (fp32, sequential fma over the rank, rounded to bf16) first.
//
// Persistent: each CTA walks row blocks (groups * RPT rows) with a grid
// stride; the raw data of the next block is loaded before the current one is
// transformed, so HBM reads overlap the arithmetic.
template <typename OutT, int S, int RPT, bool LORA>
__global__ void __launch_bounds__(kMaxThreads) rotq_rows_kernel(const RotqArgs a) {
    __shared__ float red[2][RPT][kMaxThreads / 32];
    const int G = a.G;
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int groups = blockDim.x / G;
    const int64_t chunks = a.K >> 3;
    const int64_t rows_per_block = (int64_t)groups * RPT;
    const int64_t nblocks = (a.rows + rows_per_block - 1) / rows_per_block;
    const uint16_t *x = static_cast<const uint16_t *>(a.x);
    const int wpg = G >> 5;

    Raw8 raw[RPT][S];
    auto fetch = [&](int64_t blk) {
        const int64_t row0 = (blk * groups + g) * RPT;
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int64_t c = (int64_t)s * G + t;
                const int64_t row = row0 + r;
                if (c < chunks && row < a.rows && CR_SPAN(row * a.ldx + 8 * c, 8, (a.rows - 1) * a.ldx + a.K))
                    raw[r][s].load(x + row * a.ldx + 8 * c);
                else
                    raw[r][s].zero();
            }
        }
    };

    int par = 0;
    int64_t blk = blockIdx.x;
    if (blk < nblocks) fetch(blk);
    for (; blk < nblocks; blk += gridDim.x, par ^= 1) {
        const int64_t row0 = (blk * groups + g) * RPT;
        float e[RPT][S][8];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int s = 0; s < S; ++s) raw[r][s].unpack(e[r][s]);
        if (blk + gridDim.x < nblocks) fetch(blk + gridDim.x);

        if constexpr (LORA) {
            // W' = bf16(W + coef * sum_j B[n,j] A[j,k]) with d accumulated by
            // fused multiply-adds in j order (voxprint-model-forge MOSS page:
            // merge W + scale * (alpha / rank) * B @ A before quantizing).
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int64_t c = (int64_t)s * G + t;
                if (c >= chunks) continue;
                float d[RPT][8];
#pragma unroll
                for (int r = 0; r < RPT; ++r)
#pragma unroll
                    for (int i = 0; i < 8; ++i) d[r][i] = 0.f;
#pragma unroll 4
                for (int j = 0; j < a.rank; ++j) {
                    const float4 *ap = reinterpret_cast<const float4 *>(a.lora_A + (int64_t)j * a.K + 8 * c);
                    const bool a_ok = CR_SPAN((int64_t)j * a.K + 8 * c, 8, (int64_t)a.rank * a.K);
                    float4 a0 = a_ok ? __ldg(ap) : make_float4(0.f, 0.f, 0.f, 0.f);
                    float4 a1 = a_ok ? __ldg(ap + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                    float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                    for (int r = 0; r < RPT; ++r) {
                        const int64_t row = min(row0 + r, a.rows - 1);
                        const float bj = CR_SPAN(row * a.rank + j, 1, a.rows * a.rank) ? __ldg(a.lora_B + row * a.rank + j) : 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) d[r][i] = __fmaf_rn(bj, av[i], d[r][i]);
                    }
                }
#pragma unroll
                for (int r = 0; r < RPT; ++r)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        e[r][s][i] =
                            __bfloat162float(__float2bfloat16_rn(__fmaf_rn(a.coef, d[r][i], e[r][s][i])));
            }
        }

        float amax[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            amax[r] = 0.f;
#pragma unroll
            for (int s = 0; s < S; ++s) {
                fwht8(e[r][s]);
                fwht_lanes(e[r][s], a.lanes, lane);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax[r] = maxv(amax[r], absv(e[r][s][i]));
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) amax[r] = maxv(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], m));
            if (lane == 0) red[par][r][warp] = amax[r];
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            float m = 0.f;
            for (int w = 0; w < wpg; ++w) m = maxv(m, red[par][r][g * wpg + w]);
            amax[r] = m;
        }

#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int64_t row = row0 + r;
            if (row >= a.rows) continue;
            // The code decision is taken in fp32 on the fp32-rounded transform.
            const float amax_f = amax[r];
            const float inv = amax_f > 0.f ? __fdiv_rn(127.f, amax_f) : 0.f;
            // scale = amax_u / (127 sqrt(b)), in fp32
            if (t == 0 && CR_SPAN(row, 1, a.rows)) a.scale[row] = __fdiv_rn(amax_f, a.scale_denom);
            OutT *qrow = static_cast<OutT *>(a.q) + row * a.K;
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int64_t c = (int64_t)s * G + t;
                if (c >= chunks || !CR_SPAN(row * a.K + 8 * c, 8, a.rows * a.K)) continue;
                quant_store(e[r][s], inv, qrow + 8 * c);
            }
        }
    }
}

template <typename OutT, bool LORA>
cudaError_t launch_rotq_t(const RotqArgs &base, int64_t rows, int64_t K, cudaStream_t st) {
    RotqArgs a = base;
    const int64_t chunks = K / 8;
    int G, S;
    if (chunks <= kMaxThreads) {
        G = (int)((chunks + 31) / 32 * 32);
        S = 1;
    } else {
        G = kMaxThreads;
        const int64_t need = (chunks + kMaxThreads - 1) / kMaxThreads;
        S = need <= 2 ? 2 : need <= 4 ? 4 : 8;
    }
    a.G = G;
    const int groups = G >= 256 ? 1 : 256 / G;
    const int threads = groups * G;
    auto go = [&](auto kernel, int rpt) -> cudaError_t {
        const int64_t per_cta = (int64_t)groups * rpt;
        const int64_t nblocks = (rows + per_cta - 1) / per_cta;
        const int64_t resident = (int64_t)sm_count() * blocks_per_sm(reinterpret_cast<const void *>(kernel), threads, 0);
        const int64_t grid = nblocks < resident ? nblocks : resident;
        kernel<<<(unsigned)grid, threads, 0, st>>>(a);
        return cudaGetLastError();
    };
    // Rows held per thread group: enough independent 16-byte loads in flight
    // per SM for HBM, within the register budget of 512-thread CTAs.
    constexpr int R1 = LORA ? 4 : 2;
    constexpr int R2 = 2;
    switch (S) {
        case 1: return go(rotq_rows_kernel<OutT, 1, R1, LORA>, R1);
        case 2: return go(rotq_rows_kernel<OutT, 2, R2, LORA>, R2);
        case 4: return go(rotq_rows_kernel<OutT, 4, 1, LORA>, 1);
        default: return go(rotq_rows_kernel<OutT, 8, 1, LORA>, 1);
    }
}

// ------------------------------------------------------- embedding lookup --

// out[t] = bf16( (scale[id] * Eq[id,:]) R ).  The transform runs on the integer
// codes (exact in fp32: |sums| <= 127 * 256), then one scaling.  Persistent
// like the quantizer: each CTA walks blocks of groups * RPT tokens and
// prefetches the next block's codes while it transforms the current ones.
template <int S, int RPT>
__global__ void __launch_bounds__(kMaxThreads) emb_lookup_kernel(const int64_t *ids, int64_t n, const int8_t *Eq,
                                                                 const float *scale_e, int64_t V, int64_t D,
                                                                 int lanes, int G, float inv_sqrt_b, uint16_t *out,
                                                                 unsigned *err) {
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int groups = blockDim.x / G;
    const int64_t chunks = D >> 3;
    const int64_t per_block = (int64_t)groups * RPT;
    const int64_t nblocks = (n + per_block - 1) / per_block;

    uint2 raw[RPT][S];
    float sc[RPT];
    int64_t idv[RPT];
    auto fetch = [&](int64_t blk) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int64_t tok = (blk * groups + g) * RPT + r;
            int64_t id = -1;
            if (tok < n) id = __ldg(ids + tok);
            const bool ok = tok < n && id >= 0 && id < V;
            if (tok < n && !ok && t == 0) atomicOr(err, DEVERR_INDEX);
            idv[r] = ok ? id : -1;
            sc[r] = ok && CR_SPAN(id, 1, V) ? __ldg(scale_e + id) : 0.f;
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                const int64_t c = (int64_t)sl * G + t;
                raw[r][sl] = (ok && c < chunks && CR_SPAN(id * D + 8 * c, 8, V * D)) ? __ldcs(reinterpret_cast<const uint2 *>(Eq + id * D + 8 * c))
                                                : make_uint2(0, 0);
            }
        }
    };

    int64_t blk = blockIdx.x;
    if (blk < nblocks) fetch(blk);
    for (; blk < nblocks; blk += gridDim.x) {
        float e[RPT][S][8];
        float s_cur[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            s_cur[r] = sc[r];
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                const uint32_t w[2] = {raw[r][sl].x, raw[r][sl].y};
#pragma unroll
                for (int i = 0; i < 8; ++i) e[r][sl][i] = (float)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
            }
        }
        if (blk + gridDim.x < nblocks) fetch(blk + gridDim.x);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int64_t tok = (blk * groups + g) * RPT + r;
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                fwht8(e[r][sl]);
                fwht_lanes(e[r][sl], lanes, lane);
            }
            if (tok >= n) continue;
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                const int64_t c = (int64_t)sl * G + t;
                if (c >= chunks) continue;
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float y0 = __fmul_rn(__fmul_rn(e[r][sl][2 * i], s_cur[r]), inv_sqrt_b);
                    const float y1 = __fmul_rn(__fmul_rn(e[r][sl][2 * i + 1], s_cur[r]), inv_sqrt_b);
                    __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                    w[i] = *reinterpret_cast<uint32_t *>(&h);
                }
                if (CR_SPAN(tok * D + 8 * c, 8, n * D))
                    __stcs(reinterpret_cast<uint4 *>(out + tok * D + 8 * c), make_uint4(w[0], w[1], w[2], w[3]));
            }
        }
    }
}

__global__ void widen_i8_kernel(const int8_t *A, int64_t count8, __half *out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count8; i += (int64_t)gridDim.x * blockDim.x) {
        if (!CR_SPAN(8 * i, 8, 8 * count8)) continue;
        uint2 v = __ldg(reinterpret_cast<const uint2 *>(A) + i);
        uint32_t w[2] = {v.x, v.y};
        int q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = (int8_t)((w[k >> 2] >> (8 * (k & 3))) & 0xff);
        store_codes(out + 8 * i, q);
    }
}

int lanes_of(int block) { return block / 8; }

}  // namespace

cudaError_t launch_rotq_bf16(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int block, const float *lora_A,
                             const float *lora_B, int rank, float coef, bool out_f16, void *q, float *scale,
                             cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (lora_A == nullptr && rotq_wide_ok(x, K, ldx, q))
        return launch_rotq_wide(x, rows, K, ldx, block, out_f16, q, scale, st);
    RotqArgs a{};
    a.x = x;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.lanes = lanes_of(block);
    a.scale_denom = (float)(127.0 * sqrt((double)block));
    a.q = q;
    a.scale = scale;
    a.lora_A = lora_A;
    a.lora_B = lora_B;
    a.rank = rank;
    a.coef = coef;
    if (lora_A != nullptr) return launch_rotq_t<int8_t, true>(a, rows, K, st);
    if (out_f16) return launch_rotq_t<__half, false>(a, rows, K, st);
    return launch_rotq_t<int8_t, false>(a, rows, K, st);
}

cudaError_t launch_emb_lookup(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e, int64_t V,
                              int64_t D, int block, uint16_t *out, unsigned *err, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    if (lookup_wide_ok(Eq, D, out)) return launch_lookup_wide(ids, n, Eq, scale_e, V, D, block, out, err, st);
    const int64_t chunks = D / 8;
    int G, S;
    if (chunks <= kMaxThreads) {
        G = (int)((chunks + 31) / 32 * 32);
        S = 1;
    } else {
        G = kMaxThreads;
        const int64_t need = (chunks + kMaxThreads - 1) / kMaxThreads;
        S = need <= 2 ? 2 : need <= 4 ? 4 : 8;
    }
    const int groups = G >= 256 ? 1 : 256 / G;
    const int threads = groups * G;
    const float inv_sqrt_b = (float)(1.0 / sqrt((double)block));
    const int lanes = lanes_of(block);
    auto go = [&](auto kernel, int rpt) -> cudaError_t {
        const int64_t per_cta = (int64_t)groups * rpt;
        const int64_t nblocks = (n + per_cta - 1) / per_cta;
        const int64_t resident = (int64_t)sm_count() * blocks_per_sm(reinterpret_cast<const void *>(kernel), threads, 0);
        const int64_t grid = nblocks < resident ? nblocks : resident;
        kernel<<<(unsigned)grid, threads, 0, st>>>(ids, n, Eq, scale_e, V, D, lanes, G, inv_sqrt_b, out, err);
        return cudaGetLastError();
    };
    switch (S) {
        case 1: return go(emb_lookup_kernel<1, 4>, 4);
        case 2: return go(emb_lookup_kernel<2, 2>, 2);
        case 4: return go(emb_lookup_kernel<4, 1>, 1);
        default: return go(emb_lookup_kernel<8, 1>, 1);
    }
}

cudaError_t launch_widen_i8(const int8_t *A, int64_t count, uint16_t *out, cudaStream_t st) {
    if (count == 0) return cudaSuccess;
    const int64_t count8 = count / 8;
    const int64_t blocks = (count8 + 255) / 256;
    widen_i8_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), 256, 0, st>>>(A, count8,
                                                                                 reinterpret_cast<__half *>(out));
    return cudaGetLastError();
}

}  // namespace convrot
