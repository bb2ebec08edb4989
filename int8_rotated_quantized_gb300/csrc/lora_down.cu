// Operands of the LoRA bypass (the adapter's branch on the unrotated input,
// added before the output rounding; MOSS-Image LoRA training guide, section
// 7.1: the LoRA branch of a ConvRot layer sees the unrotated input; the
// scaling coef = scale * alpha / rank follows the voxprint-model-forge MOSS
// page's merge formula):
//   xa[m, j] = coef * sum_k x[m, k] * A[j, k]    (the down-projection)
// and the parts the GEMM's tensor cores read for the branch sum_j xa[m, j] B[n, j],
// in the GEMM's accumulator units: xa[m] / dx[m] and B[n] / dw[n], where d is
// the token's (weight row's) dequantization scale, or 1 where that scale is 0.
//
// Parts.  An fp32 value v is carried as three bf16 values hi + mid + lo (hi =
// bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid); both differences are
// exact in fp32), about 24 significant bits in all.  A row of parts holds
// 64 bf16 (128 bytes, one row of a 128-byte-swizzled operand tile): hi of
// j = 0..15 at columns 0-15, mid at 16-31, lo at 32-47, zeros at 48-63;
// j >= rank is zero.
//
// One kernel, lora_operands_kernel.  x is bf16 (exact in a bf16 operand) and
// A enters as its three parts, stacked as a [48, K] bf16 operand Ap, so
// D = x Ap^T is one M = 128, N = 48 kind::f16 GEMM whose products are exact
// and whose sums accumulate in fp32 in TMEM; xa[m, j] = coef * (D[m, j] +
// D[m, 16 + j] + D[m, 32 + j]).  A CTA takes 128 rows of x and one span of K;
// the spans of one row tile form a thread-block cluster (up to 8 CTAs).
//   - one thread streams the x tiles (16 KB, 128-byte swizzled) and the fp32
//     A tiles (16 rows x 64, 4 KB; rows past rank are filled with zeros) by
//     TMA through a 4-stage ring; two warps turn each A tile into the 6 KB Ap
//     tile (the split into parts, in the swizzled layout the MMA reads), so
//     Ap never goes through memory; one thread issues the MMAs into 48 TMEM
//     columns;
//   - the two Ap warps of every CTA first write the parts of its share of B's
//     rows (the grid has at least N / (128 spans) row tiles; those past M do
//     only that);
//   - each CTA leaves its partial D [128][48] in its shared memory, and after
//     a cluster barrier CTA r adds, for rows r * 128 / spans onwards, the
//     spans' partials in span order through distributed shared memory and
//     writes the parts of xa / dx; a second cluster barrier keeps every CTA's
//     partial alive until all have read it.
// Every mbarrier wait is bounded (a timeout is recorded in the error word and
// the kernel runs to its end, through both cluster barriers).
#include "common.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "mbar.cuh"
#include "tcgen05.cuh"

namespace convrot {
namespace {

constexpr int kDnRows = 128, kDnN = 48, kDnBK = 64, kDnStages = 4, kDnThreads = 128;
constexpr int kDnXStage = kDnRows * kDnBK * 2, kDnAStage = kDnN * kDnBK * 2;  // 16 KB, 6 KB
constexpr int kDnFStage = 16 * kDnBK * 4;                                      // 4 KB of fp32 A
constexpr int kDnOffA = kDnStages * kDnXStage;
constexpr int kDnOffF = kDnOffA + kDnStages * kDnAStage;
constexpr int kDnOffBar = kDnOffF + kDnStages * kDnFStage;
constexpr int kDnNumBars = 3 * kDnStages + 1;  // full, empty, a_full per stage; done
constexpr int kDnSmem = kDnOffBar + kDnNumBars * 8 + 16 + 1024;
constexpr int kDnTmemCols = 64;
static_assert(kDnRows * kDnN * 4 <= kDnOffA, "the partial sums reuse the x ring");
// kind::f16 instruction descriptor: D fp32, A and B bf16, K-major, N = 48, M = 128
constexpr uint32_t kIdescDn = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kDnN >> 3) << 17) |
                              ((uint32_t)(kDnRows >> 4) << 24);

struct Parts3 {
    uint16_t hi, mid, lo;
};
__device__ __forceinline__ Parts3 split3(float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    return {__bfloat16_as_ushort(hi), __bfloat16_as_ushort(mid), __bfloat16_as_ushort(__float2bfloat16_rn(r2))};
}

__device__ __forceinline__ void store_parts(uint16_t *row, int j, float v) {
    const Parts3 q = split3(v);
    row[j] = q.hi;
    row[16 + j] = q.mid;
    row[32 + j] = q.lo;
    row[48 + j] = 0;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// The Ap tile of a K block (rows j, 16 + j, 32 + j = the parts of the fp32 A
// tile's row j; the TMA filled rows past rank and columns past K with zeros)
// in 128-byte-swizzle atoms: 16-byte chunk c of row r at chunk c ^ (r & 7).
// t = 0..63: two (row j, 8-column chunk c) items.
__device__ __forceinline__ void write_ap_tile(uint8_t *dst, const float *af, int t) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int item = t + 64 * it;
        const int j = item >> 3, c = item & 7;
        float v[8];
        const float4 a = *reinterpret_cast<const float4 *>(af + j * kDnBK + 8 * c);
        const float4 b = *reinterpret_cast<const float4 *>(af + j * kDnBK + 8 * c + 4);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
        uint32_t hi[4], mid[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const Parts3 p0 = split3(v[2 * e]), p1 = split3(v[2 * e + 1]);
            hi[e] = (uint32_t)p0.hi | ((uint32_t)p1.hi << 16);
            mid[e] = (uint32_t)p0.mid | ((uint32_t)p1.mid << 16);
            lo[e] = (uint32_t)p0.lo | ((uint32_t)p1.lo << 16);
        }
        const int rows[3] = {j, 16 + j, 32 + j};
        const uint32_t *src[3] = {hi, mid, lo};
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int r = rows[q];
            *reinterpret_cast<uint4 *>(dst + r * 128 + ((c ^ (r & 7)) << 4)) =
                make_uint4(src[q][0], src[q][1], src[q][2], src[q][3]);
        }
    }
}

__global__ void __launch_bounds__(kDnThreads) lora_operands_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmAf, const float *scale_x,
    int64_t M, int64_t K, int rank,
    const float *B, const float *scale_w, int64_t N, float coef, int num_kb, int kb_per_span, uint16_t *xa_parts,
    uint16_t *b_parts, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sX = base, sA = base + kDnOffA, sF = base + kDnOffF, bars = base + kDnOffBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kDnOffBar + kDnNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int spans = (int)gridDim.y;
    const uint32_t crank = cluster_rank();  // = the span (the cluster covers the spans of one row tile)
    const int64_t m0 = (int64_t)blockIdx.x * kDnRows;
    const int kb0 = (int)blockIdx.y * kb_per_span;
    const int kb1 = min(num_kb, kb0 + kb_per_span);
    const int nkb = m0 < M && kb1 > kb0 ? kb1 - kb0 : 0;  // (row tiles past M only write B's parts)
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (kDnStages + i); };
    auto a_full = [&](int i) { return bars + 8u * (2 * kDnStages + i); };
    const uint32_t done = bars + 8u * (3 * kDnStages);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDnStages; ++i) {
            mbar_init(full(i), 3);  // the producer's expect_tx (x) + the two Ap warps
            mbar_init(empty(i), 1);
            mbar_init(a_full(i), 1);  // the producer's expect_tx (fp32 A)
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

    if (warp == 0) {
        if (lane == 0) {  // x and fp32 A tiles by TMA
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmAf) : "memory");
            int i = 0;
            for (; i < nkb; ++i) {
                const int s = i % kDnStages;
                if (!mbar_wait(empty(s), ((i / kDnStages) & 1) ^ 1, abort_flag, err)) break;
                mbar_expect_tx(a_full(s), kDnFStage);
                tma_load_2d(sF + s * kDnFStage, &tmAf, a_full(s), (kb0 + i) * kDnBK, 0);
                mbar_expect_tx(full(s), kDnXStage);
                tma_load_2d(sX + s * kDnXStage, &tmX, full(s), (kb0 + i) * kDnBK, (int)m0);
            }
            for (int j = i - 1; j >= 0 && j >= i - kDnStages; --j) {  // copies in flight land before the CTA goes on
                mbar_wait_drain(a_full(j % kDnStages), (j / kDnStages) & 1);
                mbar_wait_drain(full(j % kDnStages), (j / kDnStages) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
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
    } else {  // warps 2 and 3: this CTA's share of B's parts while the first tiles load, then the Ap tiles
        const int t = threadIdx.x - 64;
        {  // a row of B per thread: its loads all in flight at once, one 128-byte row of parts out
            const int64_t ctas = (int64_t)gridDim.x * spans;
            const int64_t cta = (int64_t)blockIdx.x * spans + blockIdx.y;
            const int64_t per = (N + ctas - 1) / ctas;  // <= 128 (the launcher's grid)
            const int64_t n1 = min(N, (cta + 1) * per);
            for (int64_t n = cta * per + t; n < n1; n += 64) {
                float bv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    bv[j] = j < rank && CR_SPAN(n * rank + j, 1, N * rank) ? __ldg(B + n * rank + j) : 0.f;
                const float sw = CR_SPAN(n, 1, N) ? __ldg(scale_w + n) : 1.f;
                const float dw = sw != 0.f ? sw : 1.f;
                uint32_t w[32];  // bf16 pairs: hi at words 0-7, mid 8-15, lo 16-23, zeros 24-31
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const Parts3 p0 = split3(__fdiv_rn(bv[j], dw)), p1 = split3(__fdiv_rn(bv[j + 1], dw));
                    w[j / 2] = (uint32_t)p0.hi | ((uint32_t)p1.hi << 16);
                    w[8 + j / 2] = (uint32_t)p0.mid | ((uint32_t)p1.mid << 16);
                    w[16 + j / 2] = (uint32_t)p0.lo | ((uint32_t)p1.lo << 16);
                    w[24 + j / 2] = 0;
                }
                if (CR_SPAN(n * kLoraPartsRow, kLoraPartsRow, N * kLoraPartsRow)) {
                    uint4 *dst = reinterpret_cast<uint4 *>(b_parts + n * kLoraPartsRow);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                }
            }
        }
        // (a_full(s) completes only after the MMAs freed stage s)
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kDnStages;
            const bool got = mbar_wait(a_full(s), (i / kDnStages) & 1, abort_flag, err);
            if (!__all_sync(0xffffffffu, got)) break;
            write_ap_tile(smem + kDnOffA + s * kDnAStage, reinterpret_cast<const float *>(smem + kDnOffF + s * kDnFStage),
                          t);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s));
        }
    }
    __syncwarp();

    // this span's partial D: thread = row of the tile (TMEM lane) -> shared memory (the x ring is idle now)
    mbar_wait_drain(done, 0);
    tc_fence_after();
    float *part = reinterpret_cast<float *>(smem);  // [128][48]
    {
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
        float4 *dst = reinterpret_cast<float4 *>(part + threadIdx.x * kDnN);
#pragma unroll
        for (int i = 0; i < kDnN / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    tc_fence_before();
    cluster_barrier();  // every span's partial is in place

    // rows crank * rpc .. + rpc - 1 of the tile: xa / dx as parts, the spans added in order
    {
        const int rpc = kDnRows / spans;
        const uint32_t part_addr = smem_u32(part);
        for (int e = threadIdx.x; e < rpc * 16; e += kDnThreads) {
            const int ml = (int)crank * rpc + (e >> 4), j = e & 15;
            const int64_t m = m0 + ml;
            if (m >= M) continue;
            const uint32_t row = part_addr + (uint32_t)(ml * kDnN) * 4u;
            float d[8][3];  // all loads in flight at once (spans <= 8)
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (s < spans) {
                    d[s][0] = ld_cluster_f32(row + 4u * j, (uint32_t)s);
                    d[s][1] = ld_cluster_f32(row + 4u * (16 + j), (uint32_t)s);
                    d[s][2] = ld_cluster_f32(row + 4u * (32 + j), (uint32_t)s);
                }
            float v = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (s < spans) v = __fadd_rn(v, __fadd_rn(__fadd_rn(d[s][0], d[s][1]), d[s][2]));
            const float sx = CR_SPAN(m, 1, M) ? __ldg(scale_x + m) : 1.f;
            if (CR_SPAN(m * kLoraPartsRow + j, 49, M * kLoraPartsRow))
                store_parts(xa_parts + m * kLoraPartsRow, j, __fdiv_rn(__fmul_rn(coef, v), sx != 0.f ? sx : 1.f));
        }
    }
    cluster_barrier();  // no CTA leaves while another still reads its partial
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kDnTmemCols) : "memory");
    }
}

}  // namespace

int lora_down_spans(int64_t M, int64_t K) {
    // about 256 CTAs in all, spans of at least 4 K blocks, at most 8 spans (the cluster size)
    const int64_t tiles = (M + kDnRows - 1) / kDnRows, nkb = (K + kDnBK - 1) / kDnBK;
    int s = 1;
    while (s < 8 && tiles * s * 2 <= 256 && nkb / (2 * s) >= 4) s *= 2;
    return s;
}

cudaError_t launch_lora_operands(const uint16_t *x, const float *scale_x, int64_t M, int64_t K, const float *A,
                                 const float *B, const float *scale_w, int64_t N, int rank, float coef,
                                 uint16_t *xa_parts, uint16_t *b_parts, unsigned *err, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmX, tmAf;  // x [M, K] bf16; A [rank, K] fp32 in boxes of 16 rows (rows past rank read as 0)
    if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)K, (uint64_t)M, kDnBK, kDnRows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmAf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A, (uint64_t)K, (uint64_t)rank, kDnBK, 16,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int spans = lora_down_spans(M, K);
    const int num_kb = (int)((K + kDnBK - 1) / kDnBK);
    const int kbs = (num_kb + spans - 1) / spans;
    e = ensure_smem_attr(reinterpret_cast<const void *>(lora_operands_kernel), kDnSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    const int64_t tiles = (M + kDnRows - 1) / kDnRows, b_tiles = (N + 128 * spans - 1) / (128 * spans);
    cfg.gridDim = dim3((unsigned)(tiles > b_tiles ? tiles : b_tiles), (unsigned)spans, 1);
    cfg.blockDim = dim3(kDnThreads, 1, 1);
    cfg.dynamicSmemBytes = kDnSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)spans;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, lora_operands_kernel, tmX, tmAf, scale_x, M, K, rank, B, scale_w, N, coef, num_kb,
                           kbs, xa_parts, b_parts, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace convrot
