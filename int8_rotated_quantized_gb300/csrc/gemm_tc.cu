// Fused int8 GEMM + dequantization epilogue for sm_103a (tcgen05 + TMA + TMEM).
//
// Computes acc[m,n] = sum_k A[m,k] * B[n,k] exactly, then either writes acc as
// int32 or y = bf16(float(acc) * (sa[m] * sb[n]) + bias[n])
// (sd-scripts PR #2461, ConvRot INT8, Summary: the int8 GEMM is fused with
// the activation rotation/quantization and a dequantization epilogue;
// MOSS-Image LoRA training guide, section 7.1).
//
// Integer arithmetic on the tensor cores of sm_103a.  The int8 MMA kind of
// tcgen05 is not available on this target, so the integer codes enter the
// kind::f16 MMA as fp16 values: every code in [-127, 127] is exact in fp16,
// every product (|p| <= 16129) is exact in fp32, and a sum of integers stays
// exact in the fp32 accumulator while every partial sum is below 2^24.  The K
// loop is therefore cut into chunks of 1024 (1024 * 16129 < 2^24): each chunk
// accumulates into its own TMEM buffer, and the epilogue warps convert the
// chunk to int32 and add it to an int32 accumulator held in registers.  The
// result is the exact int32 dot product for any codes in [-127, 127].
//
// Operands.  The MMA's M side (128 rows, the operand that must be widened)
// is the WEIGHT: its int8 codes arrive by TMA and a converter warpgroup widens
// each 128x64 tile to fp16 into a 128B-swizzled K-major buffer.  The N side
// (256 rows) is the ACTIVATION, whose codes the rotate-and-quantize kernel
// already stored as fp16: TMA brings them in the 128B-swizzled layout the MMA
// reads.  Putting the weight on the 128-row side halves the conversion work
// per MMA compared with the opposite assignment.  The accumulator is therefore
// the transposed tile (TMEM lane = weight row n, column = token m).
//
// Two kernels.  gemm_s8_tc_kernel (one persistent CTA per SM) runs the modes
// that widen the int8 weight codes inside the loop (int32 output, fused
// dequantization) and is described here; gemm_pair_kernel (clusters of two
// CTAs and the 2-SM MMA, further down) runs the modes whose weight tiles
// arrive ready: codes widened beforehand, bf16 weights, the fp32-scaled
// product, and the LoRA bypass.
//
// CTA roles of gemm_s8_tc_kernel (512 threads, 128 weight rows x 256 tokens
// per tile):
//   warp 0        TMA producer of the activation tiles (one lane)
//   warp 1        TMEM allocator and MMA issuer (one lane)
//   warp 2        TMA producer of the int8 weight tiles (one lane)
//   warp 3        idle (completes warpgroup 0 for setmaxnreg)
//   warps 4-7     int8 -> fp16 converters of the weight tiles
//   warps 8-15    epilogue: TMEM -> registers, int32 accumulation, output
// Pipelines: a 4-stage activation ring (fp16 32 KB, refilled when the MMA
// is done with a slot), a 4-stage int8 weight ring (8 KB, refilled when the
// converters are done, so weight loads and their widening run ahead of the
// MMA), a 4-stage converted-weight ring (16 KB; 4 + 4 measured 3% faster than
// 6 + 3), and two 128x256 fp32 TMEM accumulators (512 columns) alternating
// per K chunk so the epilogue drains one while the MMA fills the other.
// Every wait is bounded: on expiry the kernel records DEVERR_TIMEOUT, lets
// in-flight copies and MMAs finish, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "mbar.cuh"
#include "tcgen05.cuh"
#include "wide.cuh"

namespace convrot {
namespace {

constexpr int TW = 128, TT = 256, BK = 64;  // weight rows (MMA M), tokens (MMA N), K per stage
constexpr int XSTAGES = 4, WSTAGES = 4, CSTAGES = 4;
constexpr int CHUNK_KB = 16;  // K blocks per exact fp32 chunk: 16 * 64 = 1024
constexpr int NUM_THREADS = 512;
constexpr int W8_STAGE = TW * BK;      // 8 KB int8 weight tile (TMA)
constexpr int X_STAGE = TT * BK * 2;   // 32 KB fp16 activation tile (TMA)
constexpr int WH_STAGE = TW * BK * 2;  // 16 KB widened weight tile
// Kernel modes: integer codes with an int32 result; integer codes with the
// dequantization epilogue; bf16 operands with a bf16 result (the bf16
// backward of a frozen base: one fp32 accumulation over all of K); and the
// dequantization epilogue on weight codes that a separate pass already
// widened to fp16 (no converter in the loop, the same exact integer chunks).
constexpr int kModeS32 = 0, kModeDequant = 1, kModeBf16 = 2, kModeDequantW16 = 3;
// The widened-weight dequantization mode plus a LoRA bypass term (CTA pairs
// only): y = bf16(acc * (sx * sw) + bias + sum_j xa[m, j] B[n, j]).  The term
// joins each tile's last exact-integer chunk as one more K block on the tensor
// cores: the operands arrive divided by the output's scales (xa[m] / dx[m] and
// B[n] / dw[n], d = s, or 1 where s = 0, whose codes are all zero) as three
// bf16 parts each (hi + mid + lo = the fp32 value to about 24 bits), and the
// six products of parts whose orders add up to at most 2 accumulate in fp32
// onto the chunk's integer sum; the epilogue adds that chunk to the earlier
// chunks' sum in fp32 and scales by dx * dw.
constexpr int kModeDequantW16Lora = 4;
// Widened weight codes, exact integer chunks, and an fp32 result scaled by the
// token's scale only: P[m, n] = float(acc) * sa[m] (the second reading of the
// int8 backward rotates P afterwards).
constexpr int kModeScaleF32 = 5;
// modes whose weight tiles arrive by TMA already in the MMA's format
constexpr bool weight_direct(int mode) {
    return mode == kModeBf16 || mode == kModeDequantW16 || mode == kModeDequantW16Lora || mode == kModeScaleF32;
}

// Stages of the rings when the weight tiles arrive ready by TMA (widened-weight
// and bf16 modes).  There is no int8 ring; the space it frees is left to the
// L1 cache: deeper rings (4 + 5, 4 + 6, 5 + 4, 3 + 8) and shallower ones
// (3 + 3, 3 + 4, 4 + 3) all measured slower than 4 + 4.
constexpr int XSTAGES_D = 4, CSTAGES_D = 4;

// Shared-memory layout of one kernel mode: ring offsets and barrier indices.
template <int MODE>
struct Layout {
    static constexpr bool kDirect = weight_direct(MODE);
    static constexpr int XS = kDirect ? XSTAGES_D : XSTAGES;  // activation ring
    static constexpr int WS = kDirect ? 0 : WSTAGES;          // int8 weight ring
    static constexpr int CS = kDirect ? CSTAGES_D : CSTAGES;  // ring the MMA reads the weights from
    static constexpr int OFF_X = 0;
    static constexpr int OFF_W8 = OFF_X + XS * X_STAGE;
    static constexpr int OFF_WH = OFF_W8 + WS * W8_STAGE;
    static constexpr int OFF_BAR = OFF_WH + CS * WH_STAGE;
    // One full and one empty barrier per stage of the MMA's two operands (the
    // activation ring and the fp16 weight ring advance together): the MMA
    // thread waits once and frees a stage with one commit.  The int8 weight
    // ring of the fused-widening modes has its own pair for the converters.
    static_assert(XS == CS, "the two operand rings advance together");
    static constexpr int BAR_FULL = 0, BAR_EMPTY = XS, BAR_W_FULL = 2 * XS, BAR_W_EMPTY = BAR_W_FULL + WS,
                         BAR_ACC_FULL = BAR_W_EMPTY + WS, BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
                         BAR_DRAIN = BAR_ACC_EMPTY + 2, NUM_BARS = BAR_DRAIN + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};
constexpr int TMEM_COLS = 512;
constexpr int REGS_WG0 = 48, REGS_CONV = 80, REGS_EPI = 184;
static_assert(128 * REGS_WG0 + 128 * REGS_CONV + 256 * REGS_EPI <= 65536, "register split exceeds the launch pool");

// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B format
// (bits 7-9, 10-12: 0 = fp16, 1 = bf16), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kIdescF16 = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(TT >> 3) << 17) | ((uint32_t)(TW >> 4) << 24);
constexpr uint32_t kIdescBF16 = kIdescF16 | (1u << 7) | (1u << 10);


struct GemmArgs {
    int M, N, K;
    int group;         // tiles per raster group along the grouped dimension
    int group_weight;  // 1: groups of weight tiles sweep the token tiles; 0: the reverse
    const float *sa, *sb;
    const uint16_t *bias;
    void *out;
    unsigned *err;
    uint64_t wait_limit_ns = kWaitLimitNs;  // bound of every pipeline wait
    // Failure-path self-test only: the producer named by fault_role (0 the
    // activation producer, 1 the weight producer) issues no copy at its
    // iteration fault_skip_it, so the stage it feeds never fills and the
    // consumer's bounded wait must end the kernel.  -1 outside the self-test.
    int fault_skip_it = -1;
    int fault_role = -1;
};

// All 512 threads meet here at the end; each role reaches it from its own
// branch, so no code runs after a join of regions with different register
// budgets.
__device__ __forceinline__ void end_barrier() {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(NUM_THREADS) : "memory");
}

template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Grouped raster.  A group of `group` tiles along one dimension sweeps every
// tile of the other dimension, so the group's operand tiles stay in L2 while
// the other operand streams through once per group; odd groups sweep
// backwards and start on the tiles their predecessor read last.  The host
// picks the grouped dimension and the group size from the operand sizes.
__device__ __forceinline__ void tile_coords(int tile, int num_t, int num_w, int group, bool group_weight, int &tb,
                                            int &wb) {
    const int num_g = group_weight ? num_w : num_t;  // grouped dimension
    const int num_s = group_weight ? num_t : num_w;  // swept dimension
    const int gi = tile / (group * num_s);
    const int first = gi * group;
    const int gsize = min(num_g - first, group);
    const int in_group = tile - gi * group * num_s;
    const int g = first + in_group % gsize;
    int sw = in_group / gsize;
    if (gi & 1) sw = num_s - 1 - sw;
    tb = group_weight ? sw : g;
    wb = group_weight ? g : sw;
}

// ------------------------------------------------------------------ kernel --

// Every lane of the warp polls the barrier (a single polling lane with the
// rest parked in __syncwarp measured 2x slower); the result is made
// warp-uniform so no lane runs ahead on an abort.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err,
                                          uint64_t limit_ns) {
    const bool got = mbar_wait(bar, parity, abort_flag, err, limit_ns);
    return __all_sync(0xffffffffu, got);
}

// The epilogue's stores of one thread: weight row n, the 128 tokens m0 ..
// m0 + 127 of its column half in acc (mlim of them exist; full: all 128).
// Each store instruction of a warp writes 32 consecutive n of one row m.
template <int MODE>
__device__ __forceinline__ void epi_store(const int (&acc)[128], int n, int m0, int mlim, bool full,
                                          const GemmArgs &p) {
    // (checked builds: the column's rows m0 .. m0 + min(128, mlim) - 1 lie inside out [M, N])
    if (n < p.N && (mlim <= 0 || CR_SPAN((int64_t)m0 * p.N + n, (int64_t)((full ? 128 : mlim) - 1) * p.N + 1,
                                         (int64_t)p.M * p.N))) {
        if constexpr (MODE == kModeS32) {
            int32_t *out = static_cast<int32_t *>(p.out) + (int64_t)m0 * p.N + n;
#pragma unroll
            for (int i = 0; i < 128; ++i) {
                if (full || i < mlim) *out = acc[i];
                out += p.N;
            }
        } else if constexpr (MODE == kModeScaleF32) {
            float *out = static_cast<float *>(p.out) + (int64_t)m0 * p.N + n;
#pragma unroll
            for (int i4 = 0; i4 < 128; i4 += 4) {
                float sx[4];
                if (full) {
                    const float4 v = CR_SPAN(m0 + i4, 4, p.M) ? __ldg(reinterpret_cast<const float4 *>(p.sa + m0 + i4))
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                    sx[0] = v.x, sx[1] = v.y, sx[2] = v.z, sx[3] = v.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) sx[j] = i4 + j < mlim ? __ldg(p.sa + m0 + i4 + j) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (full || i4 + j < mlim) *out = __fmul_rn(__int2float_rn(acc[i4 + j]), sx[j]);
                    out += p.N;
                }
            }
        } else if constexpr (MODE == kModeBf16) {  // (also the bypass mode: y's fp32 bits)
            uint16_t *out = static_cast<uint16_t *>(p.out) + (int64_t)m0 * p.N + n;
#pragma unroll
            for (int i = 0; i < 128; ++i) {
                if (full || i < mlim) *out = (uint16_t)float_to_bf16_bits(__int_as_float(acc[i]));
                out += p.N;
            }
        } else {  // kModeDequant, kModeDequantW16
            uint16_t *out = static_cast<uint16_t *>(p.out) + (int64_t)m0 * p.N + n;
            const float swn = CR_SPAN(n, 1, p.N) ? __ldg(p.sb + n) : 0.f;
            const bool has_bias = p.bias != nullptr;
            const float bn = has_bias ? bf16_bits_to_float(__ldg(p.bias + n)) : 0.f;
#pragma unroll
            for (int i4 = 0; i4 < 128; i4 += 4) {
                float sx[4];
                if (full) {
                    const float4 v = CR_SPAN(m0 + i4, 4, p.M) ? __ldg(reinterpret_cast<const float4 *>(p.sa + m0 + i4))
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                    sx[0] = v.x, sx[1] = v.y, sx[2] = v.z, sx[3] = v.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) sx[j] = i4 + j < mlim ? __ldg(p.sa + m0 + i4 + j) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float y = __fmul_rn(__int2float_rn(acc[i4 + j]), __fmul_rn(sx[j], swn));
                    if (has_bias) y = __fadd_rn(y, bn);
                    if (full || i4 + j < mlim) *out = (uint16_t)float_to_bf16_bits(y);
                    out += p.N;
                }
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_s8_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const GemmArgs p) {
    using L = Layout<MODE>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sX = base + L::OFF_X, sW8 = base + L::OFF_W8, sWh = base + L::OFF_WH, sBar = base + L::OFF_BAR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::XS; ++i) {
            // the producer's expect_tx (both operands' bytes when the weight tiles
            // come ready), plus the 4 converter warps in the fused-widening modes
            mbar_init(bar(L::BAR_FULL + i), L::kDirect ? 1 : 5);
            mbar_init(bar(L::BAR_EMPTY + i), 1);  // MMA commit
        }
        for (int i = 0; i < L::WS; ++i) {
            mbar_init(bar(L::BAR_W_FULL + i), 1);
            mbar_init(bar(L::BAR_W_EMPTY + i), 4);  // 4 converter warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(L::BAR_ACC_FULL + i), 1);
            mbar_init(bar(L::BAR_ACC_EMPTY + i), 8);
        }
        mbar_init(bar(L::BAR_DRAIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // p.M = tokens (activation rows), p.N = weight rows, p.K = contraction.
    const int num_t = (p.M + TT - 1) / TT;
    const int num_w = (p.N + TW - 1) / TW;
    const int num_tiles = num_t * num_w;
    const int num_kb = (p.K + BK - 1) / BK;
    // K blocks per TMEM accumulation: exact-integer chunks, or all of K for bf16
    const int chunk_kb = MODE == kModeBf16 ? num_kb : CHUNK_KB;

    if (warp < 4) {
        regs_dec<REGS_WG0>();
        if ((warp == 0 || (warp == 2 && !L::kDirect)) && lane == 0) {
            // ---------------------------------------------------- producers
            // warp 0 streams the activation tiles and, in the modes whose weight
            // tiles arrive ready (widened codes, bf16), the weight tile of the
            // same stage onto the same barrier.  In the fused-widening modes warp
            // 2 streams the int8 weight tiles into their own ring, freed by the
            // converter warps.
            const bool is_x = warp == 0;
            const int nst = is_x ? L::XS : L::WS;
            const int full0 = is_x ? L::BAR_FULL : L::BAR_W_FULL;
            const int empty0 = is_x ? L::BAR_EMPTY : L::BAR_W_EMPTY;
            asm volatile("prefetch.tensormap [%0];" ::"l"(is_x ? &tmX : &tmW) : "memory");
            if (is_x && L::kDirect) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
            int it = 0, skipped = -1;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int tb, wb;
                tile_coords(tile, num_t, num_w, p.group, p.group_weight != 0, tb, wb);
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int s = it % nst;
                    if (!mbar_wait(bar(empty0 + s), ((it / nst) & 1) ^ 1, abort_flag, p.err, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    // self-test: the named operand's copy of this stage is never issued
                    const bool skip_x = it == p.fault_skip_it && p.fault_role == 0;
                    const bool skip_w = it == p.fault_skip_it && p.fault_role == 1;
                    if (is_x) {
                        mbar_expect_tx(bar(full0 + s), X_STAGE + (L::kDirect ? WH_STAGE : 0));
                        if (!skip_x) tma_load_2d(sX + s * X_STAGE, &tmX, bar(full0 + s), kb * BK, tb * TT);
                        if (L::kDirect && !skip_w) tma_load_2d(sWh + s * WH_STAGE, &tmW, bar(full0 + s), kb * BK, wb * TW);
                        if (skip_x || (L::kDirect && skip_w)) skipped = it;  // this stage never completes
                    } else {
                        if (skip_w) {
                            skipped = it;
                            continue;
                        }
                        mbar_expect_tx(bar(full0 + s), W8_STAGE);
                        tma_load_2d(sW8 + s * W8_STAGE, &tmW, bar(full0 + s), kb * BK, wb * TW);
                    }
                }
            }
            if (!ok || skipped >= 0) {  // let the copies already issued land before the CTA exits
                for (int j = it - 1; j >= 0 && j >= it - nst; --j)
                    if (j != skipped) mbar_wait_drain(bar(full0 + j % nst), (j / nst) & 1, p.wait_limit_ns);
            }
        } else if (warp == 1 && lane == 0) {
            // --------------------------------------------------------- MMA
            int it = 0, g = 0;
            bool ok = true;
            uint32_t dcol = 0;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int kc = kb % chunk_kb;
                    if (kc == 0) {
                        const int buf = g & 1;
                        if (!mbar_wait(bar(L::BAR_ACC_EMPTY + buf), ((g >> 1) & 1) ^ 1, abort_flag, p.err,
                                       p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        dcol = (uint32_t)(buf * TT);
                    }
                    const int s = it % L::XS;  // stage of both operands
                    if (!mbar_wait(bar(L::BAR_FULL + s), (it / L::XS) & 1, abort_flag, p.err, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = sw128_desc(sWh + s * WH_STAGE + kk * 32);
                        const uint64_t bd = sw128_desc(sX + s * X_STAGE + kk * 32);
                        umma_f16(tmem + dcol, ad, bd, MODE == kModeBf16 ? kIdescBF16 : kIdescF16,
                                 (kc > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(L::BAR_EMPTY + s));
                    if (kc == chunk_kb - 1 || kb == num_kb - 1) {
                        umma_commit(bar(L::BAR_ACC_FULL + (g & 1)));
                        ++g;
                    }
                }
            }
            // All MMAs issued by this thread have completed once this fires.
            umma_commit(bar(L::BAR_DRAIN));
            mbar_wait_drain(bar(L::BAR_DRAIN), 0, p.wait_limit_ns);
        }
        __syncwarp();
        end_barrier();
        if (warp == 1) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
        }
    } else if (warp < 8) {
        // ----------------------------------------------------------- converters
        regs_dec<REGS_CONV>();
        if constexpr (!L::kDirect) {  // nothing to widen when the weight tiles come ready
        const int ct = threadIdx.x - 128;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            for (int kb = 0; kb < num_kb; ++kb, ++it) {
                const int s = it % L::WS;
                const int c = it % L::CS;
                if (!warp_wait(bar(L::BAR_W_FULL + s), (it / L::WS) & 1, abort_flag, p.err, p.wait_limit_ns) ||
                    !warp_wait(bar(L::BAR_EMPTY + c), ((it / L::CS) & 1) ^ 1, abort_flag, p.err, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = smem + L::OFF_W8 + s * W8_STAGE;
                uint8_t *dst = smem + L::OFF_WH + c * WH_STAGE;
                // 128 rows x 64 int8 (rows of 64 bytes, no swizzle) -> 128 rows x 64 fp16
                // in 128B-swizzle atoms (8 rows x 128 bytes, 16-byte chunk j of row r at j ^ (r & 7)).
                uint4 v[(TW * BK / 16) / 128];
#pragma unroll
                for (int j = 0; j < (TW * BK / 16) / 128; ++j) {
                    const int L = j * 128 + ct;
                    v[j] = *reinterpret_cast<const uint4 *>(src + (L >> 2) * BK + (L & 3) * 16);
                }
#pragma unroll
                for (int j = 0; j < (TW * BK / 16) / 128; ++j) {
                    const int L = j * 128 + ct;
                    const int row = L >> 2;
                    const int c4 = L & 3;
                    uint32_t w[8];
                    widen4(v[j].x, w[0], w[1]);
                    widen4(v[j].y, w[2], w[3]);
                    widen4(v[j].z, w[4], w[5]);
                    widen4(v[j].w, w[6], w[7]);
                    uint8_t *atom = dst + (row >> 3) * 1024 + (row & 7) * 128;
                    const int sw = row & 7;
                    *reinterpret_cast<uint4 *>(atom + (((2 * c4) ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(atom + (((2 * c4 + 1) ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(L::BAR_W_EMPTY + s));
                    mbar_arrive(bar(L::BAR_FULL + c));  // the stage's weight operand is ready
                }
            }
        }
        }
        end_barrier();
    } else {
        // ------------------------------------------------------------- epilogue
        regs_inc<REGS_EPI>();
        const int q = warp & 3;          // TMEM lane quarter = weight rows 32q .. 32q+31
        const int h = (warp - 8) >> 2;   // token half of the 256-wide tile
        int g = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            int tb, wb;
            tile_coords(tile, num_t, num_w, p.group, p.group_weight != 0, tb, wb);
            int acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            const int nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
            for (int ch = 0; ch < nchunks; ++ch, ++g) {
                const int buf = g & 1;
                if (!warp_wait(bar(L::BAR_ACC_FULL + buf), (g >> 1) & 1, abort_flag, p.err, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * TT + h * 128);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t r[16];
                    tmem_ld16(taddr + 16 * j, r);
                    tmem_wait_ld();
                    if constexpr (MODE == kModeBf16) {  // one chunk: keep the fp32 bits
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[16 * j + i] = (int)r[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[16 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::BAR_ACC_EMPTY + buf));
            }
            if (!ok) break;
            // Thread = weight row n, registers = 128 consecutive tokens m: each
            // store instruction of the warp writes 32 consecutive n of one row m.
            const int n = wb * TW + 32 * q + lane;
            const int m0 = tb * TT + h * 128;
            const int mlim = p.M - m0;  // tokens of this column half that exist
            const bool full = mlim >= 128;
            epi_store<MODE>(acc, n, m0, mlim, full, p);
        }
        end_barrier();
    }
}


// ----------------------------------------------------------- CTA-pair GEMM --
// The modes whose weight tiles arrive ready (widened codes, bf16, the fp32-
// scaled mode) on pairs of CTAs with the 2-SM MMA.  A pair (a cluster of two
// CTAs on neighbouring SMs) computes 256 weight rows x 256 tokens: CTA r of
// the pair holds, in every slot, weight rows 128 r .. 128 r + 127 (its half
// of the MMA's A) and token rows 128 r .. 128 r + 127 (its half of B) of one K
// block of 64, so a slot is 32 KB per SM instead of 48 and six slots are in
// flight, filled and freed two at a time (a pipeline stage is two K blocks).
// The leader (r = 0) sets the stage's byte count, both CTAs' copies complete on
// the leader's barrier, the leader issues tcgen05.mma.cta_group::2 (M = 256,
// N = 256) and multicasts every commit to both CTAs; each CTA's accumulator
// holds its 128 weight rows x 256 tokens and its epilogue (the same as the
// single-CTA kernel's) stores them; the epilogue warps of both CTAs free an
// accumulator buffer on the leader's barrier.  Both CTAs take part in the
// pair's TMEM allocation and release.
namespace pair {
constexpr int STAGES = 6;                    // 16 KB + 16 KB slots per CTA (7 measured slower)
// K blocks per pipeline stage: the producer fills KSUB slots onto one barrier and the MMA thread
// waits once and commits once per stage, so the hand-off runs once per 128 of K (measured against
// once per 64: 8.5% faster in the widened-weight mode, 5% in the bf16 mode on 20480-token shapes)
constexpr int KSUB = 2, SSTAGES = STAGES / KSUB;
static_assert(STAGES % KSUB == 0 && CHUNK_KB % KSUB == 0, "stages of whole slots, chunks of whole stages");
constexpr int XH_STAGE = (TT / 2) * BK * 2;  // 16 KB: this CTA's 128 token rows
constexpr int W_STAGE = TW * BK * 2;         // 16 KB: this CTA's 128 weight rows
constexpr int STG_BYTES = 32 * 32 * 2;  // a warp's 32 tokens x 32 features of bf16 output
constexpr int OFF_X = 0, OFF_W = STAGES * XH_STAGE, OFF_STG = OFF_W + STAGES * W_STAGE,
              OFF_BAR = OFF_STG + 8 * STG_BYTES;
constexpr int BAR_FULL = 0, BAR_EMPTY = STAGES, BAR_ACC_FULL = 2 * STAGES, BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
              BAR_DRAIN = BAR_ACC_EMPTY + 2, NUM_BARS = BAR_DRAIN + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory budget");
// kind::f16 with M = 256 (the pair; bits 24-28: M >> 4) and N = 256 tokens
constexpr uint32_t kIdescPairF16 = (1u << 4) | ((uint32_t)(TT >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
constexpr uint32_t kIdescPairBF16 = kIdescPairF16 | (1u << 7) | (1u << 10);
}  // namespace pair

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// A tile into this CTA's shared memory, completing on a barrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(
            dst),
        "l"(map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on the barrier at this offset in both CTAs of the pair once the MMAs issued so far complete.
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(mask)
                 : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// The bf16-output epilogue stores of the pair kernel for a warp whose 32
// features and 128 tokens all exist: each 32-token block goes through the
// warp's 2 KB of shared memory ([token][feature], written one feature per
// lane) and leaves as 16-byte stores of 8 features of one token (a quarter of
// the store instructions of writing each value on its own; measured 1.4-2%
// faster on the forward shapes).  y = bf16(acc * (sa[m] * sb[n]) + bias[n])
// (dequantization mode) or bf16 of the fp32 bits in acc (bf16 mode).
template <int MODE>
__device__ __forceinline__ void epi_store_staged(const int (&acc)[128], int n, int m0, const GemmArgs &p, uint16_t *stg,
                                                 int lane) {
    float swn = 0.f, bn = 0.f;
    bool has_bias = false;
    if constexpr (MODE == kModeDequantW16) {
        swn = __ldg(p.sb + n);
        has_bias = p.bias != nullptr;
        bn = has_bias ? bf16_bits_to_float(__ldg(p.bias + n)) : 0.f;
    }
    const int nb = n - lane;  // the warp's first feature
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int i4 = 0; i4 < 32; i4 += 4) {
            float sx[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (MODE == kModeDequantW16) {
                const float4 v = CR_SPAN(m0 + 32 * r + i4, 4, p.M)
                                     ? __ldg(reinterpret_cast<const float4 *>(p.sa + m0 + 32 * r + i4))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                sx[0] = v.x, sx[1] = v.y, sx[2] = v.z, sx[3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float y;
                if constexpr (MODE == kModeDequantW16) {
                    y = __fmul_rn(__int2float_rn(acc[32 * r + i4 + j]), __fmul_rn(sx[j], swn));
                    if (has_bias) y = __fadd_rn(y, bn);
                } else {
                    y = __int_as_float(acc[32 * r + i4 + j]);
                }
                stg[(i4 + j) * 32 + lane] = (uint16_t)float_to_bf16_bits(y);
            }
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int row = 8 * t + (lane >> 2), c = lane & 3;  // 16 bytes: features nb + 8c .. + 7 of token row
            const int64_t off = (int64_t)(m0 + 32 * r + row) * p.N + nb + 8 * c;
            if (CR_SPAN(off, 8, (int64_t)p.M * p.N))
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + off) =
                    *reinterpret_cast<const uint4 *>(stg + row * 32 + 8 * c);
        }
        __syncwarp();
    }
}

// The bypass mode's last chunk of a tile (thread = weight row n, tokens m0 ..
// m0 + 127): TMEM holds c = that chunk's integer sum + the bypass term in
// accumulator units, L / (dx * dw); v = fl(float(acc) + c) and y = v * (dx *
// dw) + bias, left as fp32 bits in acc.  With a zero term and |acc| < 2^24
// (float(acc) exact) v = float(acc + c), so y is the plain mode's float(acc) *
// (sx * sw) + bias bit for bit (where sx or sw is 0 the codes, and so acc, are
// zero).  Writing c exactly as rint(c) + (c - rint(c)) would keep that for
// any |acc|, but its two more conversions per value cost 2% of the GEMM in
// this drain, which holds the TMEM buffer; the host runs the plain forward
// for a zero coefficient instead.  The 128 token scales come in with four
// coalesced loads and reach every lane by shuffles (a load per value measured
// 2x slower).
__device__ __forceinline__ void lora_fold_chunk(int (&acc)[128], uint32_t taddr, int n, int m0, int lane,
                                                const GemmArgs &p) {
    const float swn = n < p.N && CR_SPAN(n, 1, p.N) ? __ldg(p.sb + n) : 0.f;
    const float dw = swn != 0.f ? swn : 1.f;
    const bool has_bias = p.bias != nullptr && n < p.N;
    const float bn = has_bias ? bf16_bits_to_float(__ldg(p.bias + n)) : 0.f;
    float sxr[4];  // lane l: the scales of tokens m0 + 32 u + l
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int m = m0 + 32 * u + lane;
        sxr[u] = m < p.M && CR_SPAN(m, 1, p.M) ? __ldg(p.sa + m) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[16];
        tmem_ld16(taddr + 16 * j, r);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const int i = 16 * j + t;
            const float sxm = __shfl_sync(0xffffffffu, sxr[i >> 5], i & 31);
            const float v = __fadd_rn(__int2float_rn(acc[i]), __uint_as_float(r[t]));
            const float dx = sxm != 0.f ? sxm : 1.f;
            float y = __fmul_rn(v, __fmul_rn(dx, dw));
            if (has_bias) y = __fadd_rn(y, bn);
            acc[i] = __float_as_int(y);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmXh, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmXA, const __grid_constant__ CUtensorMap tmLB,
                     const GemmArgs p) {
    static_assert(MODE == kModeDequantW16 || MODE == kModeBf16 || MODE == kModeScaleF32 || MODE == kModeDequantW16Lora,
                  "pair modes");
    using namespace pair;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sX = base + OFF_X, sW = base + OFF_W;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return base + OFF_BAR + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar(BAR_FULL + i), 1);   // the leader's expect_tx (both CTAs' bytes)
            mbar_init(bar(BAR_EMPTY + i), 1);  // the leader's multicast commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(BAR_ACC_FULL + i), 1);    // the leader's multicast commit
            mbar_init(bar(BAR_ACC_EMPTY + i), 16);  // the 8 epilogue warps of each CTA (the leader's copy is used)
        }
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // one warp of each CTA takes part in the pair's allocation
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();  // the barriers of both CTAs are initialised and the TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int num_t = (p.M + TT - 1) / TT;
    const int num_w2 = (p.N + 2 * TW - 1) / (2 * TW);
    const int num_tiles = num_t * num_w2;
    const int num_kb = (p.K + BK - 1) / BK;
    const int nss = (num_kb + KSUB - 1) / KSUB;  // pipeline stages per tile (the last may hold one K block)
    constexpr bool kSingleChunk = MODE == kModeBf16;  // one fp32 chunk over the whole contraction
    const int chunk_kb = MODE == kModeBf16 ? num_kb : CHUNK_KB;
    // the bypass mode's extra K block per tile (tmXA / tmLB: the parts of xa / dx and
    // B / dw, 128 bytes per row); it joins the tile's last chunk
    constexpr int kExtra = MODE == kModeDequantW16Lora ? 1 : 0;

    if (warp < 4) {
        regs_dec<REGS_WG0>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------ producer
            // this CTA's token and weight halves of each stage, onto the leader's barrier
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmXh) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
            if (kExtra) {
                asm volatile("prefetch.tensormap [%0];" ::"l"(&tmXA) : "memory");
                asm volatile("prefetch.tensormap [%0];" ::"l"(&tmLB) : "memory");
            }
            int it = 0, skipped = -1;
            bool ok = true;
            for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
                int tb, wb2;
                tile_coords(tile, num_t, num_w2, p.group, p.group_weight != 0, tb, wb2);
                for (int ss = 0; ss < nss + kExtra; ++ss, ++it) {
                    const int s = it % SSTAGES;
                    if (!mbar_wait(bar(BAR_EMPTY + s), ((it / SSTAGES) & 1) ^ 1, abort_flag, p.err, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    const bool extra = kExtra && ss == nss;  // same box sizes: 128 rows x 128 bytes
                    const int kb0 = ss * KSUB, nsub = extra ? 1 : min(KSUB, num_kb - kb0);
                    if (rank == 0) mbar_expect_tx(bar(BAR_FULL + s), 2 * nsub * (XH_STAGE + W_STAGE));
                    const uint32_t full = mapa_shared(bar(BAR_FULL + s), 0);
                    // self-test: the named operand's copies of this stage are never issued
                    const bool skip_x = it == p.fault_skip_it && p.fault_role == 0;
                    const bool skip_w = it == p.fault_skip_it && p.fault_role == 1;
                    for (int u = 0; u < nsub; ++u) {
                        const int slot = s * KSUB + u;
                        if (!skip_x)
                            tma_load_2d_pair(sX + slot * XH_STAGE, extra ? &tmXA : &tmXh, full,
                                             extra ? 0 : (kb0 + u) * BK, tb * TT + (int)rank * (TT / 2));
                        if (!skip_w)
                            tma_load_2d_pair(sW + slot * W_STAGE, extra ? &tmLB : &tmW, full,
                                             extra ? 0 : (kb0 + u) * BK, (wb2 * 2 + (int)rank) * TW);
                    }
                    if (skip_x || skip_w) skipped = it;
                }
            }
            // Let the copies already issued land before the CTA exits: the leader waits on its
            // barriers (which both CTAs' copies complete on); the partner's producer left its loop
            // only after a wait that ran out, far longer than a copy in flight takes.
            if ((!ok || skipped >= 0) && rank == 0) {
                for (int j = it - 1; j >= 0 && j >= it - SSTAGES; --j)
                    if (j != skipped)
                        mbar_wait_drain(bar(BAR_FULL + j % SSTAGES), (j / SSTAGES) & 1, p.wait_limit_ns);
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ----------------------------------------------------- MMA (leader)
            int it = 0, g = 0;
            bool ok = true;
            uint32_t dcol = 0;
            constexpr uint32_t kIdesc = MODE == kModeBf16 ? kIdescPairBF16 : kIdescPairF16;
            for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
                for (int ss = 0; ss < nss + kExtra; ++ss, ++it) {
                    const bool extra = kExtra && ss == nss;
                    const int kb0 = ss * KSUB, nsub = extra ? 1 : min(KSUB, num_kb - kb0);
                    // a chunk opens at the tile's first stage and, in the integer modes, every 16 K
                    // blocks (compile-time divisors only: this loop sets the hand-off rate); the
                    // bypass block opens no chunk
                    const bool open = !extra && (kSingleChunk ? ss == 0 : kb0 % CHUNK_KB == 0);
                    if (open) {
                        const int buf = g & 1;
                        if (!mbar_wait(bar(BAR_ACC_EMPTY + buf), ((g >> 1) & 1) ^ 1, abort_flag, p.err,
                                       p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        dcol = (uint32_t)(buf * TT);
                    }
                    const int s = it % SSTAGES;
                    if (!mbar_wait(bar(BAR_FULL + s), (it / SSTAGES) & 1, abort_flag, p.err, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (extra) {
                        // parts at byte offsets 0 (hi), 32 (mid), 64 (lo) of each 128-byte row, onto
                        // the chunk's integer sum: hi*hi, hi*mid, mid*hi, hi*lo, mid*mid, lo*hi
                        const int slot = s * KSUB;
#pragma unroll
                        for (int q = 0; q < 6; ++q) {
                            const int pa = q == 2 || q == 4 ? 1 : q == 5 ? 2 : 0;  // weight side
                            const int pb = q == 1 || q == 4 ? 1 : q == 3 ? 2 : 0;  // token side
                            const uint64_t ad = sw128_desc(sW + slot * W_STAGE + pa * 32);
                            const uint64_t bd = sw128_desc(sX + slot * XH_STAGE + pb * 32);
                            umma_f16_pair(tmem + dcol, ad, bd, kIdescPairBF16, 1u);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < KSUB; ++u) {
                            if (u >= nsub) break;
                            const int slot = s * KSUB + u;
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint64_t ad = sw128_desc(sW + slot * W_STAGE + kk * 32);
                                const uint64_t bd = sw128_desc(sX + slot * XH_STAGE + kk * 32);
                                umma_f16_pair(tmem + dcol, ad, bd, kIdesc, (!open || u > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    umma_commit_both(bar(BAR_EMPTY + s));
                    // a chunk closes after its 16th K block or the tile's last stage (the bypass
                    // block, when there is one)
                    const bool close =
                        extra || (ss == nss - 1 ? !kExtra : !kSingleChunk && (kb0 + KSUB) % CHUNK_KB == 0);
                    if (close) {
                        umma_commit_both(bar(BAR_ACC_FULL + (g & 1)));
                        ++g;
                    }
                }
            }
            umma_commit_pair(bar(BAR_DRAIN));  // fires once every MMA issued above has completed
            mbar_wait_drain(bar(BAR_DRAIN), 0, p.wait_limit_ns);
        }
        __syncwarp();
        end_barrier();
    } else if (warp < 8) {
        regs_dec<REGS_CONV>();  // no widening in these modes
        end_barrier();
    } else {
        // ---------------------------------------------------------- epilogue
        regs_inc<REGS_EPI>();
        const int q = warp & 3;          // TMEM lane quarter = weight rows 32q .. 32q+31 of this CTA's half
        const int h = (warp - 8) >> 2;   // token half of the 256-wide tile
        const uint32_t acc_empty0 = mapa_shared(bar(BAR_ACC_EMPTY), 0);  // the leader's
        int g = 0;
        bool ok = true;
        for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
            int tb, wb2;
            tile_coords(tile, num_t, num_w2, p.group, p.group_weight != 0, tb, wb2);
            const int n = (wb2 * 2 + (int)rank) * TW + 32 * q + lane;  // weight row (TMEM lane)
            const int mt = tb * TT + h * 128;                            // first token of the half
            int acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            const int nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
            for (int ch = 0; ch < nchunks; ++ch, ++g) {
                const int buf = g & 1;
                if (!warp_wait(bar(BAR_ACC_FULL + buf), (g >> 1) & 1, abort_flag, p.err, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * TT + h * 128);
                if (kExtra && ch == nchunks - 1) {
                    lora_fold_chunk(acc, taddr, n, mt, lane, p);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t r[16];
                        tmem_ld16(taddr + 16 * j, r);
                        tmem_wait_ld();
                        if constexpr (MODE == kModeBf16) {  // one chunk: keep the fp32 bits
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] = (int)r[i];
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)buf);
            }
            if (!ok) break;
            const int m0 = mt;
            const int mlim = p.M - m0;
            // the bypass mode's registers hold y's fp32 bits, stored as the bf16 mode stores them
            constexpr int SMODE = MODE == kModeDequantW16Lora ? kModeBf16 : MODE;
            if ((SMODE == kModeDequantW16 || SMODE == kModeBf16) && mlim >= 128 && n - lane + 32 <= p.N)
                epi_store_staged<SMODE>(acc, n, m0, p,
                                        reinterpret_cast<uint16_t *>(smem + OFF_STG + (warp - 8) * STG_BYTES), lane);
            else
                epi_store<SMODE>(acc, n, m0, mlim, mlim >= 128, p);
        }
        end_barrier();
    }
    // both CTAs: the partner's epilogue has read its accumulator and the leader's MMAs are
    // complete before the pair releases the TMEM
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------- host --

// Raster choice.  The tiles of the grouped dimension are read from DRAM once
// if `group` of them (plus the streaming tiles of one wave) stay in L2; the
// swept operand is then read once per group.  Measured on GB300, groups whose
// tiles total more than about 32 MB no longer stay resident, so the group is
// the largest count of tiles within that budget, and the orientation with the
// smaller estimated DRAM read volume wins.
constexpr int64_t kRasterBudget = 32ll << 20;

void choose_raster(int64_t num_t, int64_t num_w, int64_t K, int64_t w_elem, int &group, int &group_weight) {
    const int64_t t_tile = (int64_t)TT * K * 2, w_tile = (int64_t)TW * K * w_elem;  // fp16/bf16 codes, int8 or bf16
    const int64_t gt = std::max<int64_t>(1, std::min<int64_t>(num_t, kRasterBudget / t_tile));
    const int64_t gw = std::max<int64_t>(1, std::min<int64_t>(num_w, kRasterBudget / w_tile));
    const int64_t reads_t = num_t * t_tile + num_w * w_tile * ((num_t + gt - 1) / gt);
    const int64_t reads_w = num_w * w_tile + num_t * t_tile * ((num_w + gw - 1) / gw);
    group_weight = reads_w < reads_t ? 1 : 0;
    group = (int)(group_weight ? gw : gt);
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap &tmX, const CUtensorMap &tmW, const GemmArgs &p, int64_t tiles,
                        cudaStream_t st) {
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    constexpr int kSmem = Layout<MODE>::SMEM_BYTES;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemm_s8_tc_kernel<MODE>), kSmem);
    if (e != cudaSuccess) return e;
    gemm_s8_tc_kernel<MODE><<<grid, NUM_THREADS, kSmem, st>>>(tmX, tmW, p);
    return cudaGetLastError();
}


// The CTA-pair kernel: clusters of two CTAs, one pair per two SMs.  A is the
// token matrix (encoded here with a box of 128 rows: each CTA loads half a tile).
// tmXA / tmLB: the bypass parts (bypass mode only; other modes pass none).
template <int MODE>
cudaError_t launch_pair(CUtensorMapDataType dt, const void *A, const CUtensorMap &tmW, GemmArgs p, cudaStream_t st,
                        const CUtensorMap *tmXA = nullptr, const CUtensorMap *tmLB = nullptr) {
    CUtensorMap tmXh;
    if (!encode_2d(&tmXh, dt, 2, A, (uint64_t)p.K, (uint64_t)p.M, BK, TT / 2, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t num_t = (p.M + TT - 1) / TT, num_w2 = (p.N + 2 * TW - 1) / (2 * TW);
    int group, group_weight;
    choose_raster(num_t, num_w2, p.K, 4, group, group_weight);  // a pair's weight tile: 256 rows x 2 bytes
    p.group = group;
    p.group_weight = group_weight;
    const int64_t tiles = num_t * num_w2;
    const int max_pairs = sm_count() / 2;
    if (max_pairs <= 0) return cudaErrorNotSupported;
    const int pairs = (int)(tiles < max_pairs ? tiles : max_pairs);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemm_pair_kernel<MODE>), pair::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<MODE>, tmXh, tmW, tmXA ? *tmXA : tmXh, tmLB ? *tmLB : tmW, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const uint16_t *A, const float *sa, const int8_t *B, const float *sb, const uint16_t *bias,
                        int64_t M, int64_t N, int64_t K, void *out, bool out_s32, unsigned *err, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmX, tmW;
    if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, (uint64_t)K, (uint64_t)M, BK, TT,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, (uint64_t)K, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int64_t num_t = (M + TT - 1) / TT, num_w = (N + TW - 1) / TW;
    int group, group_weight;
    choose_raster(num_t, num_w, K, 1, group, group_weight);
    GemmArgs p{(int)M, (int)N, (int)K, group, group_weight, sa, sb, bias, out, err};
    return out_s32 ? launch_mode<kModeS32>(tmX, tmW, p, num_t * num_w, st)
                   : launch_mode<kModeDequant>(tmX, tmW, p, num_t * num_w, st);
}

cudaError_t launch_gemm_w16(const uint16_t *A, const float *sa, const uint16_t *B16, const float *sb,
                            const uint16_t *bias, int64_t M, int64_t N, int64_t K, uint16_t *out, unsigned *err,
                            cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW;
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B16, (uint64_t)K, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmArgs p{(int)M, (int)N, (int)K, 0, 0, sa, sb, bias, out, err};  // the raster is the launcher's
    return launch_pair<kModeDequantW16>(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, tmW, p, st);
}

cudaError_t launch_gemm_w16_lora(const uint16_t *A, const float *sa, const uint16_t *B16, const float *sb,
                                 const uint16_t *bias, const uint16_t *xa_parts, const uint16_t *b_parts, int64_t M,
                                 int64_t N, int64_t K, uint16_t *out, unsigned *err, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW, tmXA, tmLB;  // parts: 128-row boxes, one CTA's half of the pair's tile
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B16, (uint64_t)K, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmXA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xa_parts, kLoraPartsRow, (uint64_t)M, BK, TT / 2,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmLB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b_parts, kLoraPartsRow, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmArgs p{(int)M, (int)N, (int)K, 0, 0, sa, sb, bias, out, err};  // the raster is the launcher's
    return launch_pair<kModeDequantW16Lora>(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, tmW, p, st, &tmXA, &tmLB);
}

cudaError_t launch_gemm_w16_scale_f32(const uint16_t *A, const float *sa, const uint16_t *B16, int64_t M, int64_t N,
                                      int64_t K, float *out, unsigned *err, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW;
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B16, (uint64_t)K, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmArgs p{(int)M, (int)N, (int)K, 0, 0, sa, nullptr, nullptr, out, err};  // the raster is the launcher's
    return launch_pair<kModeScaleF32>(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, tmW, p, st);
}

cudaError_t launch_gemm_fault_selftest(bool widened, const uint16_t *A, const float *sa, const void *B,
                                      const float *sb, int64_t M, int64_t N, int64_t K, uint16_t *out, unsigned *err,
                                      uint64_t limit_ns, int skip_it, int role, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmX, tmW;
    const bool okw = widened ? encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B, (uint64_t)K, (uint64_t)N, BK, TW,
                                         CU_TENSOR_MAP_SWIZZLE_128B)
                             : encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, (uint64_t)K, (uint64_t)N, BK, TW,
                                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!okw || !encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, (uint64_t)K, (uint64_t)M, BK, TT,
                           CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t num_t = (M + TT - 1) / TT, num_w = (N + TW - 1) / TW;
    int group, group_weight;
    choose_raster(num_t, num_w, K, widened ? 2 : 1, group, group_weight);
    GemmArgs p{(int)M, (int)N, (int)K, group, group_weight, sa, sb, nullptr, out, err};
    p.wait_limit_ns = limit_ns;
    p.fault_skip_it = skip_it;
    p.fault_role = role;
    return widened ? launch_pair<kModeDequantW16>(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, tmW, p, st)
                   : launch_mode<kModeDequant>(tmX, tmW, p, num_t * num_w, st);
}

cudaError_t launch_gemm_bf16(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K, uint16_t *out,
                             unsigned *err, cudaStream_t st) {
    if (M == 0 || N == 0) return cudaSuccess;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW;
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, (uint64_t)K, (uint64_t)N, BK, TW,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmArgs p{(int)M, (int)N, (int)K, 0, 0, nullptr, nullptr, nullptr, out, err};  // the raster is the launcher's
    return launch_pair<kModeBf16>(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, tmW, p, st);
}

}  // namespace convrot
