// Row-wise kernels with 32 consecutive elements per thread: rotate + quantize
// of bf16 rows (activations, gradients, weights, the embedding table) and the
// quantized embedding lookup.
//
// Same arithmetic as the 8-element kernels in rotq.cu (the block-diagonal
// normalised Sylvester-Hadamard rotation as a fast Walsh-Hadamard transform,
// per-row absmax scale, codes by round-to-nearest-even; MOSS-Image LoRA
// training guide, section 7.1, ConvRot INT8; sd-scripts PR #2461, Summary),
// laid out for fewer instructions per element:
//   - each thread loads its 32 elements with two coalesced 256-bit loads (a
//     warp reads 2 KB of a row per pair of instructions);
//   - butterfly stages h < min(b, 32) run inside the thread on packed fp32
//     pairs, and only log2(b / 32) stages cross lanes (2 for b = 128, instead
//     of 4 with 8 elements per thread), with the stage count fixed at compile
//     time;
//   - codes leave with one or two 256-bit stores per thread.
// The kernels are persistent and prefetch the next rows' raw data while the
// current ones are transformed.  Callers use them when the row length is a
// multiple of 32 and the pointers and row strides allow 32-byte accesses;
// rotq.cu covers the other cases.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "fwht.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "mbar.cuh"
#include "wide.cuh"

namespace convrot {
namespace {

constexpr int kThreads = 512;

struct WideArgs {
    const uint16_t *x;
    int64_t rows, K, ldx;
    int G;              // threads per row (multiple of 32, <= 512)
    float scale_denom;  // fp32(127 sqrt(b))
    void *q;            // codes, row stride K
    float *scale;
};

// One row per group of G threads, S slots of 32 elements per thread.
template <typename OutT, int S, int LOGB>
__global__ void __launch_bounds__(kThreads, S == 1 ? 2 : 1) rotq_wide_kernel(const WideArgs a) {
    __shared__ float red[2][kThreads / 32];
    const int G = a.G;
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int groups = blockDim.x / G;
    const int wpg = G >> 5;
    const int64_t chunks = a.K >> 5;
    const int64_t nblocks = (a.rows + groups - 1) / groups;

    uint32_t raw[S][16];
    auto fetch = [&](int64_t blk) {
        const int64_t row = blk * groups + g;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (c < chunks && row < a.rows && CR_SPAN(row * a.ldx + 32 * c, 32, (a.rows - 1) * a.ldx + a.K)) {
                const uint16_t *p = a.x + row * a.ldx + 32 * c;
                ld256(p, raw[s]);
                ld256(p + 16, raw[s] + 8);
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
            fwht32<LOGB>(e[s], lane);
            amax = fmaxf(amax, amax32(e[s]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[par][warp] = amax;
        __syncthreads();
        float m = 0.f;
        for (int w = 0; w < wpg; ++w) m = fmaxf(m, red[par][g * wpg + w]);
        if (row < a.rows) {
            // fp32 decision on the fp32 transform; scale = amax_u / (127 sqrt(b)).
            const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
            if (t == 0 && CR_SPAN(row, 1, a.rows)) a.scale[row] = __fdiv_rn(m, a.scale_denom);
            OutT *qrow = static_cast<OutT *>(a.q) + row * a.K;
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int64_t c = (int64_t)s * G + t;
                if (c < chunks && CR_SPAN(row * a.K + 32 * c, 32, a.rows * a.K)) store_codes32(e[s], inv, qrow + 32 * c);
            }
        }
    }
}

// The same rotate + quantize with the rows staged in shared memory by TMA,
// kStages row groups ahead of the arithmetic (the register prefetch of the
// kernel above holds one): more bytes in flight per SM at the same occupancy.
// A stage is one box of whole rows seen as 128-byte segments with the 128-byte
// swizzle, so the four 16-byte reads of a thread's 32 elements hit distinct
// bank groups across the warp.  The waits are bounded (timeout recorded in the
// error word, then the kernel carries on with what it has).
constexpr int kStages = 3;

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <typename OutT, int LOGB>
__global__ void __launch_bounds__(kThreads, 2) rotq_tma_kernel(const __grid_constant__ CUtensorMap tm, const WideArgs a,
                                                               int stage_stride, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float red[2][kThreads / 32];
    __shared__ int abort_flag;
    const uint32_t raw0 = smem_u32(smem_raw);
    const uint32_t base = (raw0 + 1023u) & ~1023u;
    const uint8_t *smem = smem_raw + (base - raw0);
    const uint32_t bars = base + kStages * stage_stride;
    const int G = a.G;
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int groups = blockDim.x / G;
    const int wpg = G >> 5;
    const int64_t chunks = a.K >> 5;
    const int segs = (int)(a.K >> 6);
    const int64_t nblocks = (a.rows + groups - 1) / groups;
    const uint32_t box_bytes = (uint32_t)(groups * a.K * 2);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) mbar_init(bars + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm) : "memory");
        for (int i = 0; i < kStages; ++i) {
            const int64_t blk = blockIdx.x + (int64_t)i * gridDim.x;
            if (blk < nblocks) {
                mbar_expect_tx(bars + 8 * i, box_bytes);
                tma_load_3d(base + i * stage_stride, &tm, bars + 8 * i, 0, 0, (int)(blk * groups));
            }
        }
    }
    __syncthreads();

    int par = 0, it = 0;
    for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x, par ^= 1, ++it) {
        const int s = it % kStages;
        const int64_t row = blk * groups + g;
        (void)mbar_wait(bars + 8 * s, (uint32_t)((it / kStages) & 1), &abort_flag, err);
        float e[32];
        if (t < chunks) {
            // 32 elements = half of segment (g, t / 2): chunks 4h .. 4h + 3, swizzled
            const int sid = g * segs + (t >> 1);
            const int h = t & 1;
            const uint8_t *seg = smem + s * stage_stride + sid * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(seg + 16 * ((4 * h + c) ^ (sid & 7)));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    e[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
                    e[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) e[i] = 0.f;
        }
        fwht32<LOGB>(e, lane);
        float amax = amax32(e);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[par][warp] = amax;
        __syncthreads();  // every thread has read stage s: it can be refilled
        if (threadIdx.x == 0) {
            const int64_t nxt = blk + (int64_t)kStages * gridDim.x;
            if (nxt < nblocks) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bars + 8 * s, box_bytes);
                tma_load_3d(base + s * stage_stride, &tm, bars + 8 * s, 0, 0, (int)(nxt * groups));
            }
        }
        float m = 0.f;
        for (int w = 0; w < wpg; ++w) m = fmaxf(m, red[par][g * wpg + w]);
        if (row < a.rows) {
            const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
            if (t == 0 && CR_SPAN(row, 1, a.rows)) a.scale[row] = __fdiv_rn(m, a.scale_denom);
            if (t < chunks && CR_SPAN(row * a.K + 32 * t, 32, a.rows * a.K))
                store_codes32(e, inv, static_cast<OutT *>(a.q) + row * a.K + 32 * t);
        }
    }
    if (abort_flag && threadIdx.x == 0) {  // a wait gave up: give copies still in flight time to land
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) {
        }
    }
}

// out[t] = bf16((scale[id] * Eq[id,:]) R): the transform of the integer codes
// is exact in fp32; one scaling after it.  The ids run one row ahead of the
// code loads, which run one row ahead of the arithmetic, so no load waits on
// the id load issued in the same iteration.
template <int S, int LOGB>
__global__ void __launch_bounds__(kThreads, S == 1 ? 2 : 1) lookup_wide_kernel(const int64_t *ids, int64_t n, const int8_t *Eq,
                                                               const float *scale_e, int64_t V, int64_t D, int G,
                                                               float inv_sqrt_b, uint16_t *out, unsigned *err) {
    const int g = threadIdx.x / G;
    const int t = threadIdx.x - g * G;
    const int lane = threadIdx.x & 31;
    const int groups = blockDim.x / G;
    const int64_t chunks = D >> 5;
    const int64_t nblocks = (n + groups - 1) / groups;

    auto load_id = [&](int64_t blk) -> int64_t {
        const int64_t tok = blk * groups + g;
        return blk < nblocks && tok < n ? __ldg(ids + tok) : int64_t(-1);
    };
    uint32_t raw[S][8];
    float sc = 0.f;
    auto fetch = [&](int64_t blk, int64_t id) {
        const int64_t tok = blk * groups + g;
        const bool ok = tok < n && id >= 0 && id < V;
        if (tok < n && !ok && t == 0) atomicOr(err, DEVERR_INDEX);
        sc = ok && CR_SPAN(id, 1, V) ? __ldg(scale_e + id) : 0.f;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (ok && c < chunks && CR_SPAN(id * D + 32 * c, 32, V * D)) {
                ld256(Eq + id * D + 32 * c, raw[s]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) raw[s][i] = 0u;
            }
        }
    };

    int64_t blk = blockIdx.x;
    int64_t id_next = load_id(blk + gridDim.x);
    if (blk < nblocks) fetch(blk, load_id(blk));
    for (; blk < nblocks; blk += gridDim.x) {
        const int64_t tok = blk * groups + g;
        float e[S][32];
#pragma unroll
        for (int s = 0; s < S; ++s)
#pragma unroll
            for (int k = 0; k < 8; ++k) codes_to_f32x4(raw[s][k], &e[s][4 * k]);
        const float s_cur = sc;
        if (blk + gridDim.x < nblocks) {
            const int64_t id = id_next;
            id_next = load_id(blk + 2 * (int64_t)gridDim.x);
            fetch(blk + gridDim.x, id);
        }
#pragma unroll
        for (int s = 0; s < S; ++s) fwht32<LOGB>(e[s], lane);
        if (tok >= n) continue;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t c = (int64_t)s * G + t;
            if (c >= chunks) continue;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float y0 = e[s][2 * i], y1 = e[s][2 * i + 1];
                mul2c(y0, y1, s_cur);  // (e * s) * (1 / sqrt(b)), two roundings per lane
                mul2c(y0, y1, inv_sqrt_b);
                __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                w[i] = *reinterpret_cast<uint32_t *>(&h);
            }
            if (!CR_SPAN(tok * D + 32 * c, 32, n * D)) continue;
            uint16_t *dst = out + tok * D + 32 * c;
            st256(dst, w);
            st256(dst + 16, w + 8);
        }
    }
}

// int8 codes -> fp16 values of the same integers: 32 codes per thread per
// step (one 256-bit load, two 256-bit stores), grid-stride.
__global__ void __launch_bounds__(kThreads) widen_codes_kernel(const int8_t *A, int64_t n32, uint16_t *out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n32; i += (int64_t)gridDim.x * blockDim.x) {
        if (!CR_SPAN(32 * i, 32, 32 * n32)) continue;
        uint32_t r[8];
        ld256(A + 32 * i, r);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) widen4(r[k], w[2 * k], w[2 * k + 1]);
        st256(out + 32 * i, w);
        st256(out + 32 * i + 16, w + 8);
    }
}

int log2_of(int b) {
    int l = 0;
    while ((1 << l) < b) ++l;
    return l;
}

void shape_for(int64_t len, int &G, int &S) {
    const int64_t chunks = len / 32;
    if (chunks <= kThreads) {
        G = (int)((chunks + 31) / 32 * 32);
        S = 1;
    } else {
        G = kThreads;
        S = 2;
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch_persistent(Kernel kernel, int threads, int64_t nblocks, cudaStream_t st, Args... args) {
    const int64_t resident = (int64_t)sm_count() * blocks_per_sm(reinterpret_cast<const void *>(kernel), threads, 0);
    const int64_t grid = nblocks < resident ? nblocks : resident;
    kernel<<<(unsigned)grid, threads, 0, st>>>(args...);
    return cudaGetLastError();
}

template <typename OutT, int S>
cudaError_t rotq_wide_dispatch(int logb, const WideArgs &a, int threads, int64_t nblocks, cudaStream_t st) {
    switch (logb) {
        case 3: return launch_persistent(rotq_wide_kernel<OutT, S, 3>, threads, nblocks, st, a);
        case 4: return launch_persistent(rotq_wide_kernel<OutT, S, 4>, threads, nblocks, st, a);
        case 5: return launch_persistent(rotq_wide_kernel<OutT, S, 5>, threads, nblocks, st, a);
        case 6: return launch_persistent(rotq_wide_kernel<OutT, S, 6>, threads, nblocks, st, a);
        case 7: return launch_persistent(rotq_wide_kernel<OutT, S, 7>, threads, nblocks, st, a);
        default: return launch_persistent(rotq_wide_kernel<OutT, S, 8>, threads, nblocks, st, a);
    }
}

template <int S>
cudaError_t lookup_wide_dispatch(int logb, int threads, int64_t nblocks, cudaStream_t st, const int64_t *ids,
                                 int64_t n, const int8_t *Eq, const float *scale_e, int64_t V, int64_t D, int G,
                                 float inv_sqrt_b, uint16_t *out, unsigned *err) {
    switch (logb) {
        case 3: return launch_persistent(lookup_wide_kernel<S, 3>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
        case 4: return launch_persistent(lookup_wide_kernel<S, 4>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
        case 5: return launch_persistent(lookup_wide_kernel<S, 5>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
        case 6: return launch_persistent(lookup_wide_kernel<S, 6>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
        case 7: return launch_persistent(lookup_wide_kernel<S, 7>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
        default: return launch_persistent(lookup_wide_kernel<S, 8>, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
    }
}

bool a32(const void *p) { return ((uintptr_t)p & 31u) == 0; }

// Rows of a bf16 matrix [rows, K] (row stride ldx elements) as 64-element,
// 128-byte segments: dims {64, K/64, rows}, a box of whole rows, 128-byte
// swizzle (16-byte chunk j of segment s lands at j ^ (s & 7)).  The driver's
// encoder is looked up once.
bool encode_row_segments(CUtensorMap *map, const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (encode == nullptr || K % 64 != 0 || K / 64 > 256 || box_rows < 1 || box_rows > 256) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)(K / 64), (cuuint64_t)rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)ldx * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)(K / 64), (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows go through the TMA-staged kernel when they can be described as whole
// 128-byte segments in one box (a multiple of 64 elements, at most 16384) and
// are long: measured on GB300, the staging gains 3.5% on rows of 16384
// (236 -> 228 us for dY [20480, 16384]), nothing on rows of 4096 with fp16 codes
// and loses 5-9% on rows of 4096 with int8 codes.
constexpr int64_t kStageTmaMinRow = 8192;

template <typename OutT>
cudaError_t rotq_tma_dispatch(int logb, const CUtensorMap &tm, const WideArgs &a, int threads, int64_t nblocks,
                              int stage_stride, unsigned *err, cudaStream_t st) {
    const int smem = kStages * stage_stride + 1024 + 8 * kStages;
    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kernel), smem);
        if (e != cudaSuccess) return e;
        const int64_t resident =
            (int64_t)sm_count() * blocks_per_sm(reinterpret_cast<const void *>(kernel), threads, (size_t)smem);
        const int64_t grid = nblocks < resident ? nblocks : resident;
        kernel<<<(unsigned)grid, threads, smem, st>>>(tm, a, stage_stride, err);
        return cudaGetLastError();
    };
    switch (logb) {
        case 3: return go(rotq_tma_kernel<OutT, 3>);
        case 4: return go(rotq_tma_kernel<OutT, 4>);
        case 5: return go(rotq_tma_kernel<OutT, 5>);
        case 6: return go(rotq_tma_kernel<OutT, 6>);
        case 7: return go(rotq_tma_kernel<OutT, 7>);
        default: return go(rotq_tma_kernel<OutT, 8>);
    }
}

}  // namespace

bool rotq_wide_ok(const void *x, int64_t K, int64_t ldx, const void *q) {
    return K % 32 == 0 && K <= 32 * 2 * kThreads && ldx % 16 == 0 && a32(x) && a32(q);
}

cudaError_t launch_rotq_wide(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int block, bool out_f16, void *q,
                             float *scale, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    WideArgs a{};
    a.x = x;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.scale_denom = (float)(127.0 * sqrt((double)block));
    a.q = q;
    a.scale = scale;
    int G, S;
    shape_for(K, G, S);
    a.G = G;
    const int groups = G >= kThreads ? 1 : kThreads / G;
    const int threads = groups * G;
    const int64_t nblocks = (rows + groups - 1) / groups;
    const int logb = log2_of(block);
    unsigned *err = K >= kStageTmaMinRow ? current_error_word() : nullptr;
    if (S == 1 && K % 64 == 0 && K >= kStageTmaMinRow && K <= 16384 && err != nullptr) {
        CUtensorMap tm;
        if (encode_row_segments(&tm, x, rows, K, ldx, groups)) {
            const int stage_stride = (int)((groups * K * 2 + 1023) / 1024 * 1024);
            return out_f16 ? rotq_tma_dispatch<__half>(logb, tm, a, threads, nblocks, stage_stride, err, st)
                           : rotq_tma_dispatch<int8_t>(logb, tm, a, threads, nblocks, stage_stride, err, st);
        }
    }
    if (out_f16)
        return S == 1 ? rotq_wide_dispatch<__half, 1>(logb, a, threads, nblocks, st)
                      : rotq_wide_dispatch<__half, 2>(logb, a, threads, nblocks, st);
    return S == 1 ? rotq_wide_dispatch<int8_t, 1>(logb, a, threads, nblocks, st)
                  : rotq_wide_dispatch<int8_t, 2>(logb, a, threads, nblocks, st);
}

cudaError_t launch_widen_codes(const int8_t *A, int64_t count, uint16_t *out, cudaStream_t st) {
    if (count == 0) return cudaSuccess;
    if (count % 32 != 0 || !a32(A) || !a32(out)) return launch_widen_i8(A, count, out, st);
    const int64_t n32 = count / 32;
    const int sms = sm_count();
    const int64_t want = (n32 + kThreads - 1) / kThreads;
    const int64_t grid = want < (int64_t)sms * 4 ? want : (int64_t)sms * 4;
    widen_codes_kernel<<<(unsigned)grid, kThreads, 0, st>>>(A, n32, out);
    return cudaGetLastError();
}

bool lookup_wide_ok(const void *Eq, int64_t D, const void *out) {
    return D % 32 == 0 && D <= 32 * 2 * kThreads && a32(Eq) && a32(out);
}

cudaError_t launch_lookup_wide(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e, int64_t V,
                               int64_t D, int block, uint16_t *out, unsigned *err, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int G, S;
    shape_for(D, G, S);
    const int groups = G >= kThreads ? 1 : kThreads / G;
    const int threads = groups * G;
    const int64_t nblocks = (n + groups - 1) / groups;
    const float inv_sqrt_b = (float)(1.0 / sqrt((double)block));
    const int logb = log2_of(block);
    return S == 1 ? lookup_wide_dispatch<1>(logb, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err)
                  : lookup_wide_dispatch<2>(logb, threads, nblocks, st, ids, n, Eq, scale_e, V, D, G, inv_sqrt_b, out, err);
}

}  // namespace convrot
