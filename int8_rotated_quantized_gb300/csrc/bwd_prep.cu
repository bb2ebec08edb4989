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
#include "mbar.cuh"
#include "tcgen05.cuh"
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


// --------------------------------- bf16-mode backward weight on tensor cores --

// For b <= 128 the transform runs on the tensor cores.  Per tile of 128 weight
// rows n x 128 columns k: U^T = Hd . Q^T, Hd = blockdiag(H_b) (128 x 128,
// entries 0 and +-1, exact in fp16) and Q the tile's int8 codes as fp16
// values; the products and the sums (|u| <= 127 * 128 < 2^24) are exact in the
// fp32 accumulator, so U is the same exact integer transform as the butterflies
// of dequant_t_kernel, and the rounding that follows is that kernel's.
// Roles (512 threads, one CTA per SM, persistent over the tiles):
//   warp 0 lane 0   the int8 tiles by TMA into a 3-stage ring (128 rows x 128 bytes,
//                   128B swizzle);
//   warp 1          allocates TMEM; lane 0 issues the 8 MMAs of a tile (M = 128
//                   columns k, N = 128 rows n, K = 128) into one of two 128-column
//                   accumulators, with Hd read from TMEM (written once at the start by
//                   warps 8-11), so that only the codes are read from shared memory;
//   warps 4-7       widen the int8 tiles to fp16 in the MMA's 128B-swizzled layout
//                   (2-stage ring), 32 rows per warp;
//   warps 8-15      one TMEM lane (column k) per thread and 64 of the tile's rows n
//                   per warp (two warps per lane quarter): read the 64 values u[n]
//                   (two 32-column TMEM loads, one wait), round s_n u / sqrt(b) to
//                   bf16 (fast path, exact double-float fallback near a midpoint),
//                   stage the warp's 32 x 64 block of the [k][n] tile in shared
//                   memory (128B swizzle) and store it by TMA (clipped at the
//                   matrix edges).
// Warps of one role never wait on each other; every wait is bounded.
namespace tcdq {
constexpr int kT = 128;
constexpr int kThreads = 512;
constexpr int kQ8Stages = 3, kQ16Stages = 2;
constexpr int kQ8Bytes = kT * kT;       // int8 tile, rows of 128 bytes
constexpr int kQ16Bytes = kT * kT * 2;  // fp16 tile: 2 atoms of 128 rows x 128 bytes (64 columns each)
constexpr int kOutBytes = kT * kT * 2;  // bf16 [k][n] tile: 2 boxes of 128 rows x 64 n
constexpr int OFF_Q8 = 0;
constexpr int OFF_Q16 = OFF_Q8 + kQ8Stages * kQ8Bytes;
constexpr int OFF_OUT = OFF_Q16 + kQ16Stages * kQ16Bytes;
constexpr int OFF_SC = OFF_OUT + 2 * kOutBytes;  // per epilogue warp: [2 buffers][sh, sl][64] floats
constexpr int OFF_BAR = OFF_SC + 8 * 2 * 2 * 64 * 4;
constexpr int B_Q8F = 0, B_Q8E = kQ8Stages, B_Q16F = 2 * kQ8Stages, B_Q16E = B_Q16F + kQ16Stages,
              B_ACCF = B_Q16E + kQ16Stages, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2, NBARS = B_DRAIN + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
static_assert(SMEM <= 227 * 1024, "shared memory budget");
// TMEM columns: two 128-column accumulators, then Hd (128 lanes = rows, 64 columns of fp16 pairs)
constexpr int kTmemCols = 512, kTmemH = 2 * kT;
// kind::f16: D fp32, A and B fp16, both K-major, N = 128 (bits 17-22: N >> 3), M = 128 (bits 24-28: M >> 4)
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kT >> 3) << 17) | ((uint32_t)(kT >> 4) << 24);
}  // namespace tcdq

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}

// D += A . B with A (M = 128 rows, 16 fp16 of K per row in 8 columns) in tensor memory
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive columns of this warp's 32 TMEM lanes from 32 registers per thread
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

template <int B>
__global__ void __launch_bounds__(tcdq::kThreads, 1)
    dequant_t_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmT,
                        const float *scale_w, int N, int K, float ch, float cl, unsigned *err) {
    using namespace tcdq;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    auto bar = [&](int i) -> uint32_t { return base + OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile t = (weight rows n0 = (t / ntk) * 128, columns k0 = (t % ntk) * 128): the k blocks of a
    // row block are consecutive, so the CTAs running at one time read whole rows of Wq
    const int ntn = (N + kT - 1) / kT, ntk = (K + kT - 1) / kT;
    const int tiles = ntn * ntk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQ8Stages; ++i) {
            mbar_init(bar(B_Q8F + i), 1);
            mbar_init(bar(B_Q8E + i), 4);  // the 4 widening warps
        }
        for (int i = 0; i < kQ16Stages; ++i) {
            mbar_init(bar(B_Q16F + i), 4);
            mbar_init(bar(B_Q16E + i), 1);  // MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_ACCF + i), 1);
            mbar_init(bar(B_ACCE + i), 8);  // the 8 epilogue warps
        }
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp >= 8 && warp < 12) {
        // Hd[r][c] = H_b[r mod b][c mod b] within a diagonal block, else 0: row r = TMEM lane r, the
        // pair c = 2i, 2i + 1 in column i (low half first); warp 8 + q writes lanes 32q .. 32q + 31
        const int r = 32 * (warp & 3) + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                uint32_t pair = 0;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 64 * h + 2 * i + e;
                    const uint32_t v = (r / B) != (c / B) ? 0u : (__popc(r & c & (B - 1)) & 1) ? 0xBC00u : 0x3C00u;
                    pair |= v << (16 * e);
                }
                w[i] = pair;
            }
            tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(kTmemH + 32 * h), w);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();  // Hd is in TMEM before the first MMA
    tc_fence_after();

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------ producer
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmQ) : "memory");
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
                const int s = it % kQ8Stages;
                if (!mbar_wait(bar(B_Q8E + s), ((it / kQ8Stages) & 1) ^ 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(bar(B_Q8F + s), kQ8Bytes);
                tma_load_2d(base + OFF_Q8 + s * kQ8Bytes, &tmQ, bar(B_Q8F + s), (t % ntk) * kT, (t / ntk) * kT);
            }
            if (!ok)  // let the copies already issued land before the CTA exits
                for (int j = it - 1; j >= 0 && j >= it - kQ8Stages; --j)
                    mbar_wait_drain(bar(B_Q8F + j % kQ8Stages), (j / kQ8Stages) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ----------------------------------------------- MMA
            int it = 0;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
                const int c = it % kQ16Stages, buf = it & 1;
                if (!mbar_wait(bar(B_ACCE + buf), ((it >> 1) & 1) ^ 1, abort_flag, err) ||
                    !mbar_wait(bar(B_Q16F + c), (it / kQ16Stages) & 1, abort_flag, err))
                    break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kT / 16; ++ks) {
                    const uint32_t off = (uint32_t)((ks >> 2) * (kT * 128) + (ks & 3) * 32);
                    umma_f16_tmem_a(tmem + (uint32_t)(buf * kT), tmem + (uint32_t)(kTmemH + 8 * ks),
                                    sw128_desc(base + OFF_Q16 + c * kQ16Bytes + off), kIdesc, ks > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_Q16E + c));
                umma_commit(bar(B_ACCF + buf));
            }
            umma_commit(bar(B_DRAIN));  // fires once every MMA issued above has completed
            mbar_wait_drain(bar(B_DRAIN), 0);
        }
    } else if (warp >= 4 && warp < 8) {  // ------------------------------- widening
        const int cw = warp - 4;           // rows 32 cw .. 32 cw + 31 of each tile
        // Load j of a lane: row 32 cw + 8 (j / 2) + rsub, codes 16 c16 .. 16 c16 + 15.  Each group of 8
        // lanes takes 4 chunks of two rows whose positions mod 8 differ by xor 5, so its 16-byte reads of
        // the swizzled int8 stage and its 16-byte fp16 writes each fall on 8 distinct bank groups.
        const int rsub = (lane >> 3) ^ (((lane >> 2) & 1) * 5), csub = lane & 3;
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int s = it % kQ8Stages, c = it % kQ16Stages;
            if (!warp_wait_b(bar(B_Q8F + s), (it / kQ8Stages) & 1, abort_flag, err)) break;
            // this warp's 32 rows: 32 x 8 groups of 16 codes, 8 per lane, into registers; the stage is then free
            const uint8_t *src = smem + OFF_Q8 + s * kQ8Bytes;
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = 32 * cw + 8 * (j >> 1) + rsub, c16 = 4 * (j & 1) + csub;
                v[j] = *reinterpret_cast<const uint4 *>(src + r * 128 + ((c16 ^ (r & 7)) << 4));
            }
            // The stage goes back to the TMA (an async-proxy write) only after these loads are performed:
            // the fence depends on every loaded word and orders the generic accesses before the async ones.
            // (Without it, with the codes resident in L2, the next copy could land in the stage before
            // some lanes' loads were performed, and those lanes widened a row of a later tile.)
            uint32_t dep = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) dep ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
            asm volatile("fence.proxy.async.shared::cta;" ::"r"(dep) : "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q8E + s));
            if (!warp_wait_b(bar(B_Q16E + c), ((it / kQ16Stages) & 1) ^ 1, abort_flag, err)) break;
            uint8_t *dst = smem + OFF_Q16 + c * kQ16Bytes;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = 32 * cw + 8 * (j >> 1) + rsub;
                uint32_t w[8];
                widen4(v[j].x, w[0], w[1]);
                widen4(v[j].y, w[2], w[3]);
                widen4(v[j].z, w[4], w[5]);
                widen4(v[j].w, w[6], w[7]);
                uint8_t *row = dst + (j & 1) * (kT * 128) + r * 128;  // 64-column atom j & 1
                const int jj = 2 * csub;
                *reinterpret_cast<uint4 *>(row + ((jj ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(row + (((jj + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q16F + c));
        }
    } else if (warp >= 8) {  // -------------------------------------------- epilogue
        const int q = warp & 3;            // TMEM lanes 32q .. 32q + 31 = tile columns k
        const int half = (warp - 8) >> 2;  // tile rows n = 64 half .. 64 half + 63
        const int kl = 32 * q + lane;      // this thread's column of the tile (row of T)
        float *sc = reinterpret_cast<float *>(smem + OFF_SC) + (warp - 8) * (2 * 2 * 64);
        // the scales of this warp's 64 rows, loaded one tile ahead (2 per lane)
        auto load_scales = [&](int tt, float (&v)[2]) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = (tt / ntk) * kT + 64 * half + lane + 32 * j;
                v[j] = tt < tiles && n < N && CR_SPAN(n, 1, N) ? __ldg(scale_w + n) : 0.f;
            }
        };
        float sv_next[2];
        load_scales(blockIdx.x, sv_next);
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int buf = it & 1;
            const int n0 = (t / ntk) * kT + 64 * half, k0 = (t % ntk) * kT;
            // the row factors s_n / sqrt(B) of this warp's 64 rows as double-floats (sh + sl)
            float *sh = sc + buf * (2 * 64), *sl = sh + 64;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int nl = lane + 32 * j;
                const float sv = sv_next[j];
                const float h = __fmul_rn(sv, ch);
                sh[nl] = h;
                sl[nl] = __fmaf_rn(sv, cl, __fmaf_rn(sv, ch, -h));
            }
            load_scales(t + gridDim.x, sv_next);
            // the staging block of this buffer: the store issued from it two tiles ago has read it
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            __syncwarp();
            if (!warp_wait_b(bar(B_ACCF + buf), (it >> 1) & 1, abort_flag, err)) break;
            tc_fence_after();
            uint32_t rr[64];
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kT + 64 * half);
            tmem_ld32(taddr, rr);
            tmem_ld32(taddr + 32, rr + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_ACCE + buf));  // the accumulator is in registers
            uint8_t *row = smem + OFF_OUT + buf * kOutBytes + half * (kT * 128) + kl * 128;
#pragma unroll
            for (int g = 0; g < 8; ++g) {  // values u[n], n = 8g .. 8g + 7 of this warp's rows
                const float4 f0 = *reinterpret_cast<const float4 *>(sh + 8 * g);
                const float4 f1 = *reinterpret_cast<const float4 *>(sh + 8 * g + 4);
                const float sv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                uint32_t pk[4];
                uint32_t near = ~0u;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float p0 = __uint_as_float(rr[8 * g + 2 * i]), p1 = __uint_as_float(rr[8 * g + 2 * i + 1]);
                    mul2v(p0, p1, sv[2 * i], sv[2 * i + 1]);
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                    pk[i] = *reinterpret_cast<const uint32_t *>(&hb);
                    // low halves within 2.5 fp32 steps of a bf16 midpoint (as in dequant_t_kernel)
                    const uint32_t d = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x5410) - 0x7ffc7ffcu;
                    asm("min.u16x2 %0, %0, %1;" : "+r"(near) : "r"(d));
                }
                if ((near & 0xffffu) <= 8u || (near >> 16) <= 8u) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float u = __uint_as_float(rr[8 * g + i]);
                        const float h = sv[i], l = sl[8 * g + i];
                        const float hi = __fmul_rn(u, h);
                        const float lo = __fmaf_rn(u, l, __fmaf_rn(u, h, -hi));
                        float rh, rlo;
                        fast_two_sum(hi, lo, rh, rlo);
                        const uint32_t b = df_to_bf16(rh, rlo);
                        pk[i >> 1] = (i & 1) ? ((pk[i >> 1] & 0xffffu) | (b << 16)) : ((pk[i >> 1] & 0xffff0000u) | b);
                    }
                }
                // 16-byte chunk g of row kl in this warp's box (128B swizzle)
                *reinterpret_cast<uint4 *>(row + ((g ^ (kl & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            // this warp's 32 rows x 64 n out by TMA
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmT, base + OFF_OUT + buf * kOutBytes + half * (kT * 128) + 32 * q * 128, n0,
                             k0 + 32 * q);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    __syncwarp();  // lanes of the single-thread roles rejoin their warps before the barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

template <int B>
cudaError_t launch_dequant_t_tc(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, float ch, float cl,
                                uint16_t *T, unsigned *err, cudaStream_t st) {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap tmQ, tmT;
    if (!encode_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, (uint64_t)K, (uint64_t)N, tcdq::kT, tcdq::kT,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, (uint64_t)N, (uint64_t)K, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t tiles = ((N + tcdq::kT - 1) / tcdq::kT) * ((K + tcdq::kT - 1) / tcdq::kT);
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    e = ensure_smem_attr(reinterpret_cast<const void *>(dequant_t_tc_kernel<B>), tcdq::SMEM);
    if (e != cudaSuccess) return e;
    dequant_t_tc_kernel<B><<<grid, tcdq::kThreads, tcdq::SMEM, st>>>(tmQ, tmT, scale_w, (int)N, (int)K, ch, cl, err);
    return cudaGetLastError();
}

cudaError_t launch_dequant_t(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, uint16_t *T,
                             unsigned *err, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const double c = 1.0 / sqrt((double)block);
    const float ch = (float)c;
    const float cl = (float)(c - (double)ch);
    switch (block) {  // b <= 128 on the tensor cores (b = 256 by the butterfly kernel below)
        case 8: return launch_dequant_t_tc<8>(Wq, scale_w, N, K, ch, cl, T, err, st);
        case 16: return launch_dequant_t_tc<16>(Wq, scale_w, N, K, ch, cl, T, err, st);
        case 32: return launch_dequant_t_tc<32>(Wq, scale_w, N, K, ch, cl, T, err, st);
        case 64: return launch_dequant_t_tc<64>(Wq, scale_w, N, K, ch, cl, T, err, st);
        case 128: return launch_dequant_t_tc<128>(Wq, scale_w, N, K, ch, cl, T, err, st);
        default: break;
    }
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
