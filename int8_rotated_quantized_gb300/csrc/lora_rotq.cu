// Fused LoRA merge + rotate + quantize of weight rows, with each row split
// along K over the CTAs of a thread-block cluster.
//
// Computes, per weight row n, exactly what the merge and the quantizer define
// (voxprint-model-forge MOSS page: the LoRA pair is merged as
// W + scale * (alpha / rank) * B @ A; sd-scripts PR #2461, Summary: the merge
// happens before the ConvRot quantization; MOSS-Image LoRA training guide,
// section 7.1: block-diagonal Hadamard rotation and per-row absmax int8):
//   d[k]  = sum over j of B[n,j] * A[j,k], fused multiply-adds in j order,
//   W'[k] = bf16(coef * d[k] + W[n,k]) (one fused multiply-add, fp32),
//   u     = the unnormalised Walsh-Hadamard transform of W' on blocks of b,
//   codes = rne(u * fp32(127 / max|u|)), scale = max|u| / fp32(127 sqrt(b)).
// Every value is bit-identical to the 8-element kernel in rotq.cu.
//
// Layout for GB300.  The merge is 2 * rank fp32 operations per element, so
// the kernel keeps A in registers: thread t of CTA c owns the 4 columns
// c * KS + 4t .. + 3 and holds A[0..rank-1] at those columns (rank <= 16, 64
// registers) for the whole launch (KS / 4 threads per CTA).  A row of K columns therefore spans
// CS = K / KS CTAs, launched as one cluster.  Per tile of 8 rows:
//   1. one thread streams the CTA's 8 row slices of W into shared memory with
//      bulk copies (double-buffered, completion on an mbarrier, bounded wait);
//   2. merge: each thread computes its 4 columns of the 8 rows with packed
//      fp32x2 fused multiply-adds (B[n,j] broadcast from shared memory) and
//      writes W' as bf16 into a tile whose 16-byte pieces are xor-swizzled;
//   3. rotate: the thread that owns 32 consecutive elements of one row reads
//      them (conflict-free thanks to the swizzle), transforms them in
//      registers and across lanes, and reduces the row maximum of its CTA's
//      slice in shared memory;
//   4. the CTAs of the cluster exchange their 8 slice maxima through
//      distributed shared memory and one cluster barrier;
//   5. every CTA writes the codes of its slice; CTA 0 writes the scales.
// All CTAs of a cluster run the same tiles in the same order, so the cluster
// barrier is always reached by every thread of the cluster.  The mbarrier
// wait is bounded: on expiry the kernel records a timeout in the error word
// and carries on with the data it has, so it always returns.
#include "common.cuh"
#include "fwht.cuh"
#include "internal.h"
#include "launch_cache.h"
#include "mbar.cuh"
#include "wide.cuh"

namespace convrot {
namespace {

constexpr int kLoraMaxRank = 16;
constexpr int kRowsPerTile = 8;
constexpr int kMaxCluster = 8;

struct LoraArgs {
    const uint16_t *W;
    int64_t rows, K, ldw;
    const float *A;  // [rank, K]
    const float *B;  // [rows, rank]
    int rank;
    float coef;
    int KS;             // columns per CTA
    float scale_denom;  // fp32(127 sqrt(b))
    int8_t *q;          // [rows, K]
    float *scale;       // [rows]
    unsigned *err;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}

// 16 bytes into the shared memory of another CTA of the cluster; the bytes
// count down the transaction count of that CTA's mbarrier when they land.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint32_t remote_bar, uint4 v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// d <- b * a + d on packed fp32 pairs, one rounding per lane.
__device__ __forceinline__ void ffma2(uint64_t &d, uint64_t b, uint64_t a) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(b), "l"(a));
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Physical 16-byte piece of logical piece P in a row of the merged tile:
// pieces 4c .. 4c + 3 (the 32 elements of chunk c) are permuted by
// (c >> 1) & 3, so the 8 lanes of a quarter warp that read the same piece of
// 8 consecutive chunks hit 8 different bank groups.
__device__ __forceinline__ int swz(int P) { return (P & ~3) | ((P ^ (P >> 3)) & 3); }

struct LoraSmem {
    // dynamic layout: win[2][8][KS] bf16 | wp[8][KS] bf16 | then this struct
    float xch[2][kMaxCluster][kRowsPerTile];    // slice maxima received from each CTA
    uint64_t bp[2][kRowsPerTile][kLoraMaxRank];  // (B[n,j], B[n,j]) of a tile's rows
    int rowmax[2][kRowsPerTile];                // this CTA's slice maxima (fp32 bits)
    unsigned long long bar[2];                  // W slices landed
    unsigned long long xbar[2];                 // all CTAs' maxima landed
    int abort_flag;
};

// RB: the rank rounded up to 4, 8 or 16.  Terms j >= rank run with A = B = 0:
// adding the exact product +0 to d leaves every d bit-identical (d starts at
// +0 and can never be -0), so the merge equals the rank-term sum.
template <int LOGB, int RB>
__global__ void __launch_bounds__(512, 1) lora_rotq_kernel(const LoraArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int KS = a.KS;
    uint16_t *win = reinterpret_cast<uint16_t *>(smem);
    uint16_t *wp = win + 2 * kRowsPerTile * KS;
    LoraSmem &sh = *reinterpret_cast<LoraSmem *>(wp + kRowsPerTile * KS);
    const int t = threadIdx.x;
    const int lane = t & 31;
    const uint32_t crank = cluster_rank();
    const int csize = gridDim.x;
    const int64_t k0 = (int64_t)crank * KS;
    const int64_t ntiles = (a.rows + kRowsPerTile - 1) / kRowsPerTile;
    const uint32_t slice_bytes = (uint32_t)KS * 2;

    if (t < 2 * kRowsPerTile) (&sh.rowmax[0][0])[t] = 0;
    if (t == 0) {
        sh.abort_flag = 0;
        mbar_init(smem_u32(&sh.bar[0]), 1);
        mbar_init(smem_u32(&sh.bar[1]), 1);
        mbar_init(smem_u32(&sh.xbar[0]), 1);
        mbar_init(smem_u32(&sh.xbar[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int64_t tile, int buf) {
        const int64_t r0 = tile * kRowsPerTile;
        const int64_t left = a.rows - r0;
        const int nr = left < kRowsPerTile ? (int)left : kRowsPerTile;
        const uint32_t bar = smem_u32(&sh.bar[buf]);
        mbar_expect_tx(bar, slice_bytes * nr);
        for (int r = 0; r < nr; ++r)  // (checked builds: a skipped copy leaves the barrier to its bounded wait)
            if (CR_SPAN((r0 + r) * a.ldw + k0, KS, (a.rows - 1) * a.ldw + a.K))
                bulk_load(smem_u32(win + (buf * kRowsPerTile + r) * KS), a.W + (r0 + r) * a.ldw + k0, slice_bytes, bar);
    };
    const int64_t stride = gridDim.y;
    int64_t tile = blockIdx.y;
    if (t == 0) {
        if (tile < ntiles) issue(tile, 0);
        if (tile + stride < ntiles) issue(tile + stride, 1);
    }

    // A[j, k0 + 4t .. + 3] for every j as two packed pairs, held for the whole launch.
    uint64_t av[RB][2];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
        ulonglong2 v = make_ulonglong2(0ull, 0ull);
        if (j < a.rank && CR_SPAN((int64_t)j * a.K + k0 + 4 * t, 4, (int64_t)a.rank * a.K)) v = __ldg(reinterpret_cast<const ulonglong2 *>(a.A + (int64_t)j * a.K + k0 + 4 * t));
        av[j][0] = v.x, av[j][1] = v.y;
    }
    const uint64_t cc = pack2(a.coef, a.coef);

    // Phase-2 ownership: 32 consecutive elements (chunk c) of tile row `prow`.
    const int cpr = KS >> 5;  // chunks per row slice
    const int prow = t / cpr;
    const int pc = t - prow * cpr;
    const int seg = cpr < 32 ? cpr : 32;  // lanes of one row within a warp
    const int P1 = t >> 1;                // phase-1 piece holding columns 4t .. 4t + 3
    uint16_t *wdst = wp + 8 * swz(P1) + 4 * (t & 1);

    // B of a tile's rows, duplicated into fp32 pairs (zero for j >= rank).
    auto fill_b = [&](int64_t tl, int pb) {
        const int64_t r0 = tl * kRowsPerTile;
        for (int i = t; i < kRowsPerTile * RB; i += blockDim.x) {
            const int r = i / RB, j = i - r * RB;
            const int64_t br = r0 + r < a.rows ? r0 + r : a.rows - 1;
            const float bv = j < a.rank && CR_SPAN(br * a.rank + j, 1, a.rows * a.rank) ? __ldg(a.B + br * a.rank + j) : 0.f;
            sh.bp[pb][r][j] = pack2(bv, bv);
        }
    };
    if (tile < ntiles) fill_b(tile, 0);

    cluster_sync();  // every CTA of the cluster has initialised its barriers before any remote store

    // Two CTA barriers per tile: B (merged tile complete) and C (slice maxima
    // complete).  Buffers indexed by `buf` alternate between tiles.
    bool ok = true;
    for (int it = 0; tile < ntiles; tile += stride, ++it) {
        const int buf = it & 1;
        const int64_t r0 = tile * kRowsPerTile;
        if (t == 0) mbar_expect_tx(smem_u32(&sh.xbar[buf]), 4 * kRowsPerTile * csize);
        if (!mbar_wait(smem_u32(&sh.bar[buf]), (it >> 1) & 1, &sh.abort_flag, a.err)) ok = false;

        // ---- merge: 4 columns x 8 rows per thread -> swizzled bf16 tile
        const uint16_t *wsrc = win + buf * kRowsPerTile * KS + 4 * t;
#pragma unroll 4
        for (int r = 0; r < kRowsPerTile; ++r) {
            uint64_t d01 = 0ull, d23 = 0ull;
#pragma unroll
            for (int j = 0; j < RB; j += 2) {
                const ulonglong2 b2 = *reinterpret_cast<const ulonglong2 *>(&sh.bp[buf][r][j]);
                ffma2(d01, b2.x, av[j][0]);
                ffma2(d23, b2.x, av[j][1]);
                ffma2(d01, b2.y, av[j + 1][0]);
                ffma2(d23, b2.y, av[j + 1][1]);
            }
            const uint2 wr = *reinterpret_cast<const uint2 *>(wsrc + r * KS);
            uint64_t w01 = pack2(__uint_as_float(wr.x << 16), __uint_as_float(wr.x & 0xffff0000u));
            uint64_t w23 = pack2(__uint_as_float(wr.y << 16), __uint_as_float(wr.y & 0xffff0000u));
            ffma2(w01, cc, d01);  // coef * d + w
            ffma2(w23, cc, d23);
            float f0, f1, f2, f3;
            unpack2(w01, f0, f1);
            unpack2(w23, f2, f3);
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(f0, f1);
            const __nv_bfloat162 h23 = __floats2bfloat162_rn(f2, f3);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t *>(&h01);
            o.y = *reinterpret_cast<const uint32_t *>(&h23);
            *reinterpret_cast<uint2 *>(wdst + r * KS) = o;
        }
        __syncthreads();  // B: merged tile complete; win[buf] and bp[buf] consumed
        if (t == 0 && tile + 2 * stride < ntiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(tile + 2 * stride, buf);
        }
        // rowmax[buf ^ 1] was last read by the sends of the previous tile, which precede B
        if (t < kRowsPerTile) sh.rowmax[buf ^ 1][t] = 0;
        if (tile + stride < ntiles) fill_b(tile + stride, buf ^ 1);  // read after C

        // ---- rotate the slice of row prow and reduce its maximum
        float e[32];
        {
            uint32_t raw[16];
            const uint16_t *src = wp + prow * KS;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint4 v = *reinterpret_cast<const uint4 *>(src + 8 * swz(4 * pc + p));
                raw[4 * p] = v.x, raw[4 * p + 1] = v.y, raw[4 * p + 2] = v.z, raw[4 * p + 3] = v.w;
            }
            unpack_bf16x32(raw, e);
        }
        fwht32<LOGB>(e, lane);
        float m = amax32(e);
        for (int s = 1; s < seg; s <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
        if ((lane & (seg - 1)) == 0) atomicMax(&sh.rowmax[buf][prow], __float_as_int(m));
        __syncthreads();  // C
        // send this CTA's 8 slice maxima to every CTA of the cluster (itself included)
        for (int i = t; i < 2 * csize; i += blockDim.x) {
            const int peer = i >> 1, h = i & 1;
            const uint4 v = *reinterpret_cast<const uint4 *>(&sh.rowmax[buf][4 * h]);
            st_async_v4(map_to(smem_u32(&sh.xch[buf][crank][4 * h]), (uint32_t)peer),
                        map_to(smem_u32(&sh.xbar[buf]), (uint32_t)peer), v);
        }
        if (!mbar_wait(smem_u32(&sh.xbar[buf]), (it >> 1) & 1, &sh.abort_flag, a.err)) ok = false;

        // ---- codes of this slice, scales from CTA 0
        float mx = 0.f;
        for (int q = 0; q < csize; ++q) mx = fmaxf(mx, sh.xch[buf][q][prow]);
        const int64_t row = r0 + prow;
        if (row < a.rows) {
            const float inv = mx > 0.f ? __fdiv_rn(127.f, mx) : 0.f;
            if (CR_SPAN(row * a.K + k0 + 32 * pc, 32, a.rows * a.K)) store_codes32(e, inv, a.q + row * a.K + k0 + 32 * pc);
            if (crank == 0 && pc == 0 && CR_SPAN(row, 1, a.rows)) a.scale[row] = __fdiv_rn(mx, a.scale_denom);
        }
    }
    if (!ok) {  // a wait gave up: let the copies already issued land before the CTA exits
        for (int i = 0; i < 2; ++i) {
            mbar_wait_drain(smem_u32(&sh.bar[i]), 0);
            mbar_wait_drain(smem_u32(&sh.bar[i]), 1);
            mbar_wait_drain(smem_u32(&sh.xbar[i]), 0);
            mbar_wait_drain(smem_u32(&sh.xbar[i]), 1);
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

int log2_of(int b) {
    int l = 0;
    while ((1 << l) < b) ++l;
    return l;
}

// Columns per CTA: a power of two from 128 to 2048 (a multiple of the block)
// that splits K over at most 8 CTAs; 512 or less is preferred (128 threads,
// up to four CTAs per SM, whose phases overlap).  0 if there is none.
int64_t slice_of(int64_t K, int block) {
    for (int64_t limit : {512, 2048})
        for (int cs = 1; cs <= kMaxCluster; ++cs) {
            if (K % cs) continue;
            const int64_t ks = K / cs;
            if (ks <= limit && ks >= 128 && (ks & (ks - 1)) == 0 && ks % block == 0) return ks;
        }
    return 0;
}

size_t smem_bytes(int64_t KS) { return (size_t)3 * kRowsPerTile * KS * 2 + sizeof(LoraSmem); }

template <int LOGB, int RB>
cudaError_t launch_lora_t(const LoraArgs &a, int cs, cudaStream_t st) {
    auto kernel = lora_rotq_kernel<LOGB, RB>;
    const size_t sm = smem_bytes(a.KS);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kernel), (int)sm);
    if (e != cudaSuccess) return e;
    const int threads = (int)(a.KS / 4);
    const int64_t ntiles = (a.rows + kRowsPerTile - 1) / kRowsPerTile;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(cs, 1, 1);
    // resident clusters of this configuration, queried once per device and shape
    static std::map<std::tuple<int, int, size_t>, int> cluster_cache;
    static std::mutex cluster_mu;
    int clusters = 0;
    {
        std::lock_guard<std::mutex> lock(cluster_mu);
        const auto key = std::make_tuple(current_device(), cs, sm);
        auto it = cluster_cache.find(key);
        if (it != cluster_cache.end()) {
            clusters = it->second;
        } else {
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters <= 0) {
                (void)cudaGetLastError();
                const int sms = sm_count();
                clusters = sms / cs > 0 ? sms / cs : 1;
            }
            cluster_cache[key] = clusters;
        }
    }
    cfg.gridDim = dim3(cs, (unsigned)(ntiles < clusters ? ntiles : clusters), 1);
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int RB>
cudaError_t launch_lora_rb(const LoraArgs &a, int cs, int logb, cudaStream_t st) {
    switch (logb) {
        case 3: return launch_lora_t<3, RB>(a, cs, st);
        case 4: return launch_lora_t<4, RB>(a, cs, st);
        case 5: return launch_lora_t<5, RB>(a, cs, st);
        case 6: return launch_lora_t<6, RB>(a, cs, st);
        case 7: return launch_lora_t<7, RB>(a, cs, st);
        default: return launch_lora_t<8, RB>(a, cs, st);
    }
}

}  // namespace

bool lora_cluster_ok(const void *W, int64_t K, int64_t ldw, int block, const float *A, int rank, const void *q) {
    if (rank < 1 || rank > kLoraMaxRank || block > 256) return false;
    if (slice_of(K, block) == 0) return false;
    return ((uintptr_t)W & 15u) == 0 && (ldw % 8) == 0 && ((uintptr_t)A & 15u) == 0 && ((uintptr_t)q & 31u) == 0;
}

cudaError_t launch_lora_cluster(const uint16_t *W, int64_t rows, int64_t K, int64_t ldw, int block, const float *A,
                                const float *B, int rank, float coef, int8_t *q, float *scale, unsigned *err,
                                cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    LoraArgs a{};
    a.W = W;
    a.rows = rows;
    a.K = K;
    a.ldw = ldw;
    a.A = A;
    a.B = B;
    a.rank = rank;
    a.coef = coef;
    a.KS = (int)slice_of(K, block);
    a.scale_denom = (float)(127.0 * sqrt((double)block));
    a.q = q;
    a.scale = scale;
    a.err = err;
    const int cs = (int)(K / a.KS);
    if (rank <= 4) return launch_lora_rb<4>(a, cs, log2_of(block), st);
    if (rank <= 8) return launch_lora_rb<8>(a, cs, log2_of(block), st);
    return launch_lora_rb<16>(a, cs, log2_of(block), st);
}

}  // namespace convrot
