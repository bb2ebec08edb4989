// Operands of the LoRA bypass (the adapter's branch on the unrotated input,
// added before the output rounding; MOSS-Image LoRA training guide, section
// 7.1: the LoRA branch of a ConvRot layer sees the unrotated input; the
// scaling coef = scale * alpha / rank follows the voxprint-model-forge MOSS
// page's merge formula):
//   xa[m, j] = coef * sum_k x[m, k] * A[j, k]    (the down-projection)
// and the parts the GEMM's tensor cores read for the branch sum_j xa[m, j] B[n, j].
//
// Parts.  An fp32 value v is carried as three bf16 values hi + mid + lo (hi =
// bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid); both differences are
// exact in fp32), about 24 significant bits in all.  A row of parts holds
// 64 bf16 (128 bytes, one row of a 128-byte-swizzled operand tile): hi of
// j = 0..15 at columns 0-15, mid at 16-31, lo at 32-47, zeros at 48-63;
// j >= rank is zero.
//
// Down-projection on the tensor cores.  x is bf16 (exact in a bf16 operand)
// and A enters as its three parts, stacked as a [48, K] bf16 matrix Ap, so
// D = x Ap^T is one M = 128, N = 48 kind::f16 GEMM whose products are exact
// and whose sums accumulate in fp32 in TMEM; xa[m, j] = coef * (D[m, j] +
// D[m, 16 + j] + D[m, 32 + j]).  A CTA takes 128 rows of x and one span of K
// (the spans split K so that enough CTAs run; each writes its fp32 D to
// part[span]); a second kernel adds the spans in order and writes the parts
// of xa.  One thread issues the TMA copies (4-stage ring of 16 KB x tiles and
// 6 KB Ap tiles, both 128-byte swizzled), one thread the MMAs; every wait is
// bounded (a timeout is recorded in the error word and the kernel finishes).
#include "common.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "mbar.cuh"
#include "tcgen05.cuh"

namespace convrot {
namespace {

constexpr int kDnRows = 128, kDnN = 48, kDnBK = 64, kDnStages = 4;
constexpr int kDnXStage = kDnRows * kDnBK * 2, kDnAStage = kDnN * kDnBK * 2;
constexpr int kDnSmem = kDnStages * (kDnXStage + kDnAStage) + 2 * kDnStages * 8 + 8 + 16 + 1024;
constexpr int kDnTmemCols = 64;
// kind::f16 instruction descriptor: D fp32, A and B bf16, K-major, N = 48, M = 128
constexpr uint32_t kIdescDn = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kDnN >> 3) << 17) |
                              ((uint32_t)(kDnRows >> 4) << 24);

__device__ __forceinline__ void store_parts(uint16_t *row, int j, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    row[j] = __bfloat16_as_ushort(hi);
    row[16 + j] = __bfloat16_as_ushort(mid);
    row[32 + j] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
    row[48 + j] = 0;
}

__global__ void __launch_bounds__(128) lora_down_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const __grid_constant__ CUtensorMap tmA, int64_t M,
                                                           int num_kb, int kb_per_span, float *part, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sX = base, sA = base + kDnStages * kDnXStage;
    const uint32_t bars = sA + kDnStages * kDnAStage;  // full[4], empty[4], done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bars - base) + (2 * kDnStages + 1) * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.x * kDnRows;
    const int kb0 = blockIdx.y * kb_per_span;
    const int kb1 = min(num_kb, kb0 + kb_per_span);
    const int nkb = kb1 > kb0 ? kb1 - kb0 : 0;
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (kDnStages + i); };
    const uint32_t done = bars + 8u * (2 * kDnStages);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDnStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kDnTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {  // TMA producer
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
        int i = 0;
        for (; i < nkb; ++i) {
            const int s = i % kDnStages;
            if (!mbar_wait(empty(s), ((i / kDnStages) & 1) ^ 1, abort_flag, err)) break;
            mbar_expect_tx(full(s), kDnXStage + kDnAStage);
            tma_load_2d(sX + s * kDnXStage, &tmX, full(s), (kb0 + i) * kDnBK, (int)m0);
            tma_load_2d(sA + s * kDnAStage, &tmA, full(s), (kb0 + i) * kDnBK, 0);
        }
        for (int j = i - 1; j >= 0 && j >= i - kDnStages; --j)  // copies in flight land before the CTA exits
            mbar_wait_drain(full(j % kDnStages), (j / kDnStages) & 1);
    } else if (warp == 1 && lane == 0) {  // MMA issuer
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kDnStages;
            if (!mbar_wait(full(s), (i / kDnStages) & 1, abort_flag, err)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kDnBK / 16; ++kk)
                umma_f16(tmem, sw128_desc(sX + s * kDnXStage + kk * 32), sw128_desc(sA + s * kDnAStage + kk * 32),
                         kIdescDn, (i > 0 || kk > 0) ? 1u : 0u);
            umma_commit(empty(s));
        }
        if (nkb > 0)
            umma_commit(done);  // fires once every MMA issued above has completed
        else
            mbar_arrive(done);
    }
    __syncwarp();
    // epilogue: thread = row m of the tile (TMEM lane), 48 columns
    mbar_wait_drain(done, 0);
    tc_fence_after();
    const int64_t m = m0 + 32 * warp + lane;
    float v[kDnN];
    if (nkb > 0) {
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int c = 0; c < kDnN / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(taddr + 16 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[16 * c + i] = __uint_as_float(r[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < kDnN; ++i) v[i] = 0.f;
    }
    if (m < M && CR_SPAN(((int64_t)blockIdx.y * M + m) * kDnN, kDnN, (int64_t)gridDim.y * M * kDnN)) {
        float4 *dst = reinterpret_cast<float4 *>(part + ((int64_t)blockIdx.y * M + m) * kDnN);
#pragma unroll
        for (int i = 0; i < kDnN / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kDnTmemCols) : "memory");
    }
}

// xa[m, j] = coef * sum over spans s (in order) of (D_s[m, j] + D_s[m, 16 + j] + D_s[m, 32 + j]), as parts.
// (One thread per (m, j): four j per thread with 16-byte loads measured slower, 5.3 -> 6.8 us.)
__global__ void lora_down_combine_kernel(const float *part, int spans, int64_t M, float coef, uint16_t *xa_parts) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < M * 16; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i >> 4;
        const int j = (int)(i & 15);
        float v = 0.f;
        for (int s = 0; s < spans; ++s) {
            const float *d = part + ((int64_t)s * M + m) * kDnN;
            if (!CR_SPAN(((int64_t)s * M + m) * kDnN + j, 33, (int64_t)spans * M * kDnN)) continue;
            v = __fadd_rn(v, __fadd_rn(__fadd_rn(d[j], d[16 + j]), d[32 + j]));
        }
        if (CR_SPAN(m * kLoraPartsRow + j, 49, M * kLoraPartsRow)) store_parts(xa_parts + m * kLoraPartsRow, j, __fmul_rn(coef, v));
    }
}

// Ap [48, K] (the parts of A's rows, j >= rank zero) and b_parts [N][64] (the parts of B's rows).
__global__ void lora_parts_kernel(const float *A, int64_t K, const float *B, int64_t N, int rank, uint16_t *ap,
                                  uint16_t *b_parts) {
    const int64_t na = 16 * K;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < na + 16 * N;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (i < na) {
            const int j = (int)(i / K);
            const int64_t k = i - (int64_t)j * K;
            const float v = j < rank && CR_SPAN((int64_t)j * K + k, 1, (int64_t)rank * K) ? A[(int64_t)j * K + k] : 0.f;
            if (!CR_SPAN((int64_t)(32 + j) * K + k, 1, 48 * K)) continue;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const float r1 = __fsub_rn(v, __bfloat162float(hi));
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const float r2 = __fsub_rn(r1, __bfloat162float(mid));
            ap[(int64_t)j * K + k] = __bfloat16_as_ushort(hi);
            ap[(int64_t)(16 + j) * K + k] = __bfloat16_as_ushort(mid);
            ap[(int64_t)(32 + j) * K + k] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
        } else {
            const int64_t t = i - na, n = t >> 4;
            const int j = (int)(t & 15);
            if (!CR_SPAN(n * kLoraPartsRow + j, 49, N * kLoraPartsRow)) continue;
            store_parts(b_parts + n * kLoraPartsRow, j, j < rank && CR_SPAN(n * rank + j, 1, N * rank) ? B[n * rank + j] : 0.f);
        }
    }
}

}  // namespace

int lora_down_spans(int64_t M, int64_t K) {
    // about 256 CTAs in all, spans of at least 4 K blocks, at most 8 spans
    const int64_t tiles = (M + kDnRows - 1) / kDnRows, nkb = (K + kDnBK - 1) / kDnBK;
    int s = 1;
    while (s < 8 && tiles * s * 2 <= 256 && nkb / (2 * s) >= 4) s *= 2;
    return s;
}

cudaError_t launch_lora_operands(const uint16_t *x, int64_t M, int64_t K, const float *A, const float *B, int64_t N,
                                 int rank, float coef, uint16_t *ap, uint16_t *xa_parts, uint16_t *b_parts,
                                 float *part, unsigned *err, cudaStream_t st) {
    if (M == 0 && N == 0) return cudaSuccess;
    const int64_t items = 16 * K + 16 * N;
    const int64_t pblocks = (items + 255) / 256 < 4096 ? (items + 255) / 256 : 4096;
    lora_parts_kernel<<<(unsigned)pblocks, 256, 0, st>>>(A, K, B, N, rank, ap, b_parts);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || M == 0) return e;
    e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmX, tmA;
    if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)K, (uint64_t)M, kDnBK, kDnRows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ap, (uint64_t)K, (uint64_t)kDnN, kDnBK, kDnN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int spans = lora_down_spans(M, K);
    const int num_kb = (int)((K + kDnBK - 1) / kDnBK);
    const int kbs = (num_kb + spans - 1) / spans;
    e = ensure_smem_attr(reinterpret_cast<const void *>(lora_down_tc_kernel), kDnSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((M + kDnRows - 1) / kDnRows), (unsigned)spans);
    lora_down_tc_kernel<<<grid, 128, kDnSmem, st>>>(tmX, tmA, M, num_kb, kbs, part, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t cblocks = (M * 16 + 255) / 256 < 4096 ? (M * 16 + 255) / 256 : 4096;
    lora_down_combine_kernel<<<(unsigned)cblocks, 256, 0, st>>>(part, spans, M, coef, xa_parts);
    return cudaGetLastError();
}

}  // namespace convrot
