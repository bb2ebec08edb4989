/*
 * convrot.h -- C ABI of libconvrot, a GB300 (sm_103a) implementation of the
 * ConvRot INT8 linear layer.
 *
 * What the layer computes (MOSS-Image LoRA training guide,
 * docs/moss_image_train_network.md, section 7.1 "VRAM Usage Optimization",
 * paragraph "ConvRot INT8"; sd-scripts pull request #2461 "ConvRot INT8",
 * Summary):
 *   - frozen base weights W[N,K] are rotated along K by a block-diagonal,
 *     normalised Sylvester-Hadamard matrix R = I (x) H_b / sqrt(b) and
 *     quantized to int8 one output row (channel) at a time, with one fp32
 *     scale per row;
 *   - at run time each activation row is rotated by the same R and quantized
 *     per row to int8 with a dynamic absmax scale;
 *   - an int8 x int8 GEMM accumulates exactly and a dequantization epilogue
 *     multiplies by scale_x[m] * scale_w[n] and writes bf16.  Because R is
 *     orthogonal, (x R)(W R)^T = x W^T;
 *   - for a frozen base only the input gradient is needed;
 *   - the token embedding table is stored the same way, so a lookup
 *     dequantizes the row and applies the inverse rotation (R is symmetric
 *     and orthogonal, hence its own inverse).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer, 16-byte aligned, row-major and
 *     contiguous unless a leading dimension is given.  bf16 and fp16 tensors
 *     are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued on it; no entry point synchronises except convrot_get_error.
 *   - The caller owns every buffer; the library allocates no device memory.
 *   - Fixed dtypes: bf16 activations/weights/outputs, int8 codes, fp32 scales.
 *     No dtype is inferred from another tensor.
 *   - Block sizes: block in {8, 16, 32, 64, 128, 256}; the rotated length must
 *     be a multiple of block and of 16, and at most CONVROT_MAX_ROW.
 *   - Argument errors are returned synchronously and nothing is enqueued.
 *     CONVROT_ERR_CUDA means a launch failed.  Errors found on the device (an
 *     out-of-range token id, a pipeline wait that exceeded its time limit) set
 *     a sticky device word that convrot_get_error() reports and clears.
 *   - Inputs must be finite.  Empty problems (M, N or n equal to 0) are valid
 *     and enqueue nothing.
 */
#ifndef CONVROT_H
#define CONVROT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CONVROT_API __attribute__((visibility("default")))
#else
#define CONVROT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONVROT_OK = 0,
    CONVROT_ERR_INVALID_ARG = 1,   /* bad size, block, alignment or null pointer */
    CONVROT_ERR_UNSUPPORTED = 2,   /* no sm_100-family GPU, or size beyond a limit */
    CONVROT_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    CONVROT_ERR_TIMEOUT = 4,       /* a device-side pipeline wait hit its limit */
    CONVROT_ERR_INDEX = 5,         /* an embedding id was outside [0, V) */
    CONVROT_ERR_BOUNDS = 6         /* checked builds only: a kernel's access left its tensor (skipped) */
} convrot_status;

/* Longest row the rotate-and-quantize kernels accept (elements). */
#define CONVROT_MAX_ROW 32768

typedef void *convrot_stream_t; /* a cudaStream_t */

/* Human-readable name of a status code (static string). */
CONVROT_API const char *convrot_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
CONVROT_API int convrot_version(void);

/* Synchronises `stream`, then reports and clears the device error word:
 * CONVROT_ERR_INDEX / CONVROT_ERR_TIMEOUT if a kernel recorded one since the
 * last call, CONVROT_ERR_CUDA if the stream itself failed, else CONVROT_OK.
 * The checked variant of the library (libconvrot_checked, built with
 * -DCONVROT_CHECKED) checks the index of the kernels' global-memory accesses
 * against their tensors' extents, skips any that falls outside, and reports
 * it here first as CONVROT_ERR_BOUNDS; the release library has no such checks. */
CONVROT_API int convrot_get_error(convrot_stream_t stream);

/* ---------------------------------------------------------------- weights -- */

/* Load-time weight quantization (guide 7.1: int8 per output channel; PR #2461
 * Summary: the base is quantized while loading, after any LoRA has been merged
 * into it; voxprint-model-forge MOSS page: the merge is W + scale*(alpha/rank)*B@A).
 *   W        bf16 [N, K], row stride ldw (elements, >= K, multiple of 8).
 *   lora_A   fp32 [rank, K] or NULL; lora_B fp32 [N, rank] or NULL (both or neither).
 *            When given, W' = bf16_rne(W + c * B@A) with c = fp32(scale*alpha/rank),
 *            evaluated in fp32 with sequential fused multiply-adds over the rank.
 *   Wq       out int8 [N, K] contiguous: codes of the rows of W' R.
 *   scale_w  out fp32 [N]: max|row of W' R| / 127 (0 for an all-zero row).
 * Row slabs (the row-chunked quantization of a large embedding table) are the
 * same call on W + row0*ldw with N = rows of the slab and lora_B + row0*rank.
 * 1 <= rank <= 64 when the LoRA pair is given. */
CONVROT_API int convrot_quantize_weight(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int block,
                            const float *lora_A, const float *lora_B, int rank, float alpha,
                            float scale, int8_t *Wq, float *scale_w, convrot_stream_t stream);

/* ------------------------------------------------------------ activations -- */

/* Online activation rotation + dynamic per-row quantization (guide 7.1; PR
 * #2461 Summary on convrot_int8_kernels.py).
 *   x        bf16 [M, K], row stride ldx (elements, >= K, multiple of 8).
 *   xq       out [M, K] contiguous: the int8 codes of x R stored as fp16 values
 *            (every code in [-127, 127] is exact in fp16; this is the operand
 *            format of the GEMM below, whose tensor-core path reads fp16).
 *   scale_x  out fp32 [M]. */
CONVROT_API int convrot_quantize_activation(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int block,
                                uint16_t *xq, float *scale_x, convrot_stream_t stream);

/* The fused int8 GEMM + dequantization epilogue on quantized operands:
 *   y[m,n] = bf16_rne( float(acc[m,n]) * (scale_x[m] * scale_w[n]) + bias[n] ),
 *   acc[m,n] = sum_k xq[m,k] * Wq[n,k]   (exact integer sum, as int32)
 *   xq       [M, K] fp16-held codes (from convrot_quantize_activation).
 *   scale_x  fp32 [M], 16-byte aligned.
 *   Wq       int8 [N, K]; scale_w fp32 [N]; bias bf16 [N] or NULL.
 *   y        out bf16 [M, N] contiguous.
 * K multiple of 16 and <= 2^17 (so |acc| < 2^31 for any codes); N multiple of 16. */
CONVROT_API int convrot_gemm_dequant(const uint16_t *xq, const float *scale_x, int64_t M, int64_t K,
                         const int8_t *Wq, const float *scale_w, int64_t N, const uint16_t *bias,
                         uint16_t *y, convrot_stream_t stream);

/* int8 codes -> fp16 values of the same integers (every code in [-127, 127]
 * is exact in fp16): the operand format of the tensor-core path, which has no
 * int8 kind on this GPU.  q int8 [count], out16 fp16 [count], both 16-byte
 * aligned; count a multiple of 16. */
CONVROT_API int convrot_widen_codes(const int8_t *q, int64_t count, uint16_t *out16, convrot_stream_t stream);

/* convrot_gemm_dequant with the weight codes already widened to fp16 values
 * (Wq16 [N, K], from convrot_widen_codes): the same exact integer accumulation
 * and epilogue, without widening inside the GEMM.  Same limits. */
CONVROT_API int convrot_gemm_dequant_w16(const uint16_t *xq, const float *scale_x, int64_t M, int64_t K,
                             const uint16_t *Wq16, const float *scale_w, int64_t N, const uint16_t *bias,
                             uint16_t *y, convrot_stream_t stream);

/* Bytes of workspace convrot_linear_fwd / convrot_linear_bwd_x need for M rows
 * of length K (the fp16-held codes and the fp32 scales). */
CONVROT_API size_t convrot_act_workspace_bytes(int64_t M, int64_t K);

/* Bytes of workspace with which convrot_linear_fwd (and convrot_linear_bwd_x
 * with N and K exchanged) takes its faster path: the activation codes and
 * scales plus a transient fp16 copy of the weight codes, [N, K] (see below). */
CONVROT_API size_t convrot_linear_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* Forward of the ConvRot INT8 linear layer (guide 7.1: online activation
 * rotation and dynamic per-row int8 quantization fused with the int8 matmul
 * and its dequantization; PR #2461 Summary on convrot_int8_kernels.py):
 * convrot_quantize_activation into `workspace`, then the int8 GEMM with the
 * dequantization epilogue.  x bf16
 * [M, K] contiguous; y bf16 [M, N]; workspace device memory of at least
 * convrot_act_workspace_bytes(M, K), 256-byte aligned.  With at least
 * convrot_linear_workspace_bytes(M, K, N) bytes the weight codes are first
 * widened into the workspace as fp16 values (convrot_widen_codes) and the GEMM
 * reads them directly (convrot_gemm_dequant_w16); the weight stays int8 at
 * rest and the result is bit-identical either way.  The workspace must not be
 * shared by calls in flight on other streams. */
CONVROT_API int convrot_linear_fwd(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq,
                       const float *scale_w, int64_t N, int block, const uint16_t *bias,
                       uint16_t *y, void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* Bytes of workspace convrot_linear_fwd_lora needs: those of the widened-weight
 * path plus the scaled down-projection and the adapter's B as three bf16 parts
 * per value (128 bytes per row of M and of N, each rounded up to 256). */
CONVROT_API size_t convrot_linear_lora_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* Forward with an unmerged LoRA adapter as a bypass (the LoRA branch of a
 * frozen ConvRot layer sees the unrotated input; guide 7.1, PR #2461 Summary;
 * the merge formula of the voxprint-model-forge MOSS page gives the scaling):
 *   y = bf16( acc * scale_x[m] * scale_w[n] + bias[n]
 *             + sum_j (coef * sum_k x[m,k] lora_A[j,k]) * lora_B[n,j] ),
 *   coef = fp32(scale * alpha / rank).  The down-projection is summed in fp32;
 *   the branch runs on the tensor cores in the GEMM's accumulator units (its
 *   factors divided by scale_x[m] and scale_w[n], 1 taking the place of a zero
 *   scale), each fp32 factor split into three bf16 parts (about 24 bits), and
 *   is accumulated in fp32 onto the last integer chunk of the product before
 *   the dequantization and the rounding.  coef = 0 runs convrot_linear_fwd
 *   (bit for bit its result).
 * x bf16 [M, K] (K multiple of 32); lora_A fp32 [rank, K] (16-byte aligned); lora_B fp32 [N, rank];
 * 1 <= rank <= 16; workspace >= convrot_linear_lora_workspace_bytes(M, K, N),
 * 256-byte aligned.  Weight codes as in convrot_linear_fwd; a weight row whose
 * scale is 0 must hold zero codes (convrot_quantize_weight writes it so), or
 * that row of y is undefined.  Branch values beyond fp32's range once divided
 * by scale_x[m] * scale_w[n] (scales near 1e-30) overflow to inf. */
CONVROT_API int convrot_linear_fwd_lora(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq,
                            const float *scale_w, int64_t N, int block, const uint16_t *bias,
                            const float *lora_A, const float *lora_B, int rank, float alpha, float scale,
                            uint16_t *y, void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* Forward without a workspace, for callers that cannot allocate device
 * memory on this path: a host framework or plugin that only passes in
 * pointers to memory it owns, a latency-critical loop where cudaMalloc (which
 * synchronises the device) is not allowed, or a process held to a fixed
 * device-memory budget.  The pages have no counterpart of this entry point;
 * it computes exactly what convrot_linear_fwd computes, with the activation
 * codes and scales kept in one fixed device array inside the library instead
 * of a caller workspace.
 *   - The array is convrot_linear_fwd_noalloc_max_bytes() bytes (64 MiB +
 *     256 KiB) on every GPU that loads the library, held until the process
 *     exits.  Problems needing more (M*K*2 + M*4 bytes, each part rounded up
 *     to 256; at K = 4096 at most M = 8219 rows) return
 *     CONVROT_ERR_UNSUPPORTED and enqueue nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  Do not use the library across a cudaDeviceReset: the
 *     cached address belongs to the context that was reset.
 *   - The GEMM of this entry point widens the int8 weight codes inside its
 *     loop (there is no workspace for a widened copy): the speed of
 *     convrot_linear_fwd with a small workspace, below that of its
 *     widened-weight path.
 *   - All calls share the array: calls whose kernels can overlap on the GPU
 *     (other streams, other host threads) race and must be serialised by the
 *     caller.  Nothing needs clearing between calls: each call rewrites all
 *     it reads.
 *   - No allocation of any kind happens inside the call.
 * Arguments, layouts and errors are those of convrot_linear_fwd without the
 * workspace. */
CONVROT_API int convrot_linear_fwd_noalloc(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq,
                               const float *scale_w, int64_t N, int block, const uint16_t *bias,
                               uint16_t *y, convrot_stream_t stream);

/* Size in bytes of the fixed device array used by convrot_linear_fwd_noalloc. */
CONVROT_API size_t convrot_linear_fwd_noalloc_max_bytes(void);

/* -------------------------------------------------------- frozen backward -- */

/* Bytes of workspace convrot_prepare_bwd_weight needs: two 32-bit words per
 * column of W_eff^T (K), cleared and used by the call. */
CONVROT_API size_t convrot_bwd_weight_workspace_bytes(int64_t N, int64_t K);

/* One-off preparation of the int8 backward weight (guide 7.1 and 4.1: the
 * opt-in int8 backward computes the input gradient with the same fused int8
 * GEMM as the forward; PR #2461 Summary: the base is frozen, so only grad_x).  The GEMM is reused
 * unchanged, so its weight operand must be a ConvRot quantization along the
 * new contraction dimension N:
 *   W_eff    = (scale_w (.) Wq) R      (the dequantized base in the original basis; every
 *              rotated value is the fp32 rounding of the exact one, decided in fp32 where it
 *              is far from a rounding boundary and in double-float arithmetic, about 48
 *              significant bits, near one)
 *   WtQ      out int8 [K, N]: codes of the rows of W_eff^T rotated along N
 *   scale_wt out fp32 [K]
 * N and K multiples of block and of 16; workspace >= convrot_bwd_weight_workspace_bytes. */
CONVROT_API int convrot_prepare_bwd_weight(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K,
                               int block, int8_t *WtQ, float *scale_wt, void *workspace,
                               size_t ws_bytes, convrot_stream_t stream);

/* Input gradient of the frozen layer through the int8 GEMM (guide 4.1 and 7.1:
 * the opt-in int8 backward reuses the fused int8 GEMM for grad_x; PR #2461
 * Summary: frozen base, so only the input gradient):
 *   dX = bf16( acc * scale_dy[m] * scale_wt[k] ),  acc = quant(dY R_N) . WtQ^T
 *   dY bf16 [M, N]; WtQ int8 [K, N]; scale_wt fp32 [K]; dX out bf16 [M, K];
 *   workspace >= convrot_act_workspace_bytes(M, N). */
CONVROT_API int convrot_linear_bwd_x(const uint16_t *dY, int64_t M, int64_t N, const int8_t *WtQ,
                         const float *scale_wt, int64_t K, int block, uint16_t *dX,
                         void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* Bytes of workspace convrot_linear_bwd_x_r2 needs: dY codes (fp16-held) and
 * scales, the transient fp16 transpose of Wq and the fp32 product [M, K]. */
CONVROT_API size_t convrot_bwd_x_r2_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Input gradient through the int8 GEMM, second reading (the pages leave the
 * operand open; this reading keeps Wq as stored and needs no prepared copy):
 *   D   = fp32(dY[m,n] * scale_w[n]);  Dq, s_d = per-row absmax codes of D, no rotation
 *   dX  = bf16( (s_d[m] * sum_n Dq[m,n] Wq[n,k]) R )   R along K in blocks of `block`
 * dY bf16 [M, N]; Wq int8 [N, K] with scale_w fp32 [N] (from convrot_quantize_weight);
 * dX out bf16 [M, K]; N and K multiples of 32 and of 16, at most 32768; dY and dX
 * 32-byte aligned; workspace >= convrot_bwd_x_r2_workspace_bytes(M, N, K), 256-byte aligned. */
CONVROT_API int convrot_linear_bwd_x_r2(const uint16_t *dY, int64_t M, int64_t N, const int8_t *Wq,
                            const float *scale_w, int64_t K, int block, uint16_t *dX,
                            void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* ------------------------------------------------- bf16 frozen backward -- */

/* The default backward mode of the layer (guide 4.1: the backward option
 * takes bf16, the default, or int8; PR #2461 Summary: frozen base, grad_x
 * only).  The base is dequantized transiently and the input gradient is a bf16
 * matmul:
 *   W_eff    = bf16_rne( (scale_w (.) Wq) R )  rounded once from a double-float
 *              value; written transposed, WeffT bf16 [K, N] contiguous.
 *   Wq int8 [N, K], scale_w fp32 [N]; N multiple of 16, K multiple of block and 16.
 * Writes only WeffT; nothing is kept between calls. */
CONVROT_API int convrot_dequant_weight_t(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K,
                             int block, uint16_t *WeffT, convrot_stream_t stream);

/* bf16 GEMM on the tensor cores: C[m,n] = bf16_rne( sum_k A[m,k] * B[n,k] ) with
 * the sum accumulated in fp32.  A bf16 [M, K], B bf16 [N, K], C out bf16 [M, N],
 * all contiguous and 16-byte aligned; K multiple of 16, N multiple of 16. */
CONVROT_API int convrot_gemm_bf16(const uint16_t *A, int64_t M, int64_t K, const uint16_t *B, int64_t N,
                      uint16_t *C, convrot_stream_t stream);

/* Bytes of workspace convrot_linear_bwd_x_bf16 needs (WeffT, bf16 [K, N]). */
CONVROT_API size_t convrot_bwd_x_bf16_workspace_bytes(int64_t N, int64_t K);

/* Input gradient of the frozen layer in bf16 mode:
 *   dX = bf16( dY . W_eff ),  W_eff as in convrot_dequant_weight_t
 *   dY bf16 [M, N]; Wq int8 [N, K]; scale_w fp32 [N]; dX out bf16 [M, K];
 *   workspace >= convrot_bwd_x_bf16_workspace_bytes(N, K), 256-byte aligned
 *   (it receives WeffT). */
CONVROT_API int convrot_linear_bwd_x_bf16(const uint16_t *dY, int64_t M, int64_t N, const int8_t *Wq,
                              const float *scale_w, int64_t K, int block, uint16_t *dX,
                              void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* -------------------------------------------------------------- embedding -- */

/* Quantized token-embedding lookup (PR #2461 Summary: the int8 text encoder
 * quantizes embed_tokens in the rotated basis, so the lookup dequantizes the
 * rows and applies the inverse rotation).
 *   ids      int64 [n]; Eq int8 [V, D]; scale_e fp32 [V]
 *   out      bf16 [n, D]: bf16_rne((scale_e[id] * Eq[id,:]) R)
 * An id outside [0, V) produces a zero row and sets CONVROT_ERR_INDEX in the
 * device error word (no out-of-bounds read). */
CONVROT_API int convrot_embedding_lookup(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e,
                             int64_t V, int64_t D, int block, uint16_t *out,
                             convrot_stream_t stream);

/* ------------------------------------------------------------- test entry -- */

/* Bytes of workspace convrot_gemm_s32 needs (A widened to fp16 codes). */
CONVROT_API size_t convrot_gemm_s32_workspace_bytes(int64_t M, int64_t K);

/* The GEMM's exact integer accumulator, for bit-exact checks:
 *   C[m,n] = sum_k A[m,k] * B[n,k] as int32, A int8 [M, K], B int8 [N, K].
 * Runs the same tensor-core kernel as convrot_gemm_dequant with an int32
 * epilogue.  Entries of A and B must lie in [-127, 127] (the codes the
 * quantizers produce).  K multiple of 16 and <= 2^17 (so |C| < 2^31). */
CONVROT_API int convrot_gemm_s32(const int8_t *A, const int8_t *B, int64_t M, int64_t N, int64_t K,
                     int32_t *C, void *workspace, size_t ws_bytes, convrot_stream_t stream);

/* Test entry for the failure path: launches one CTA that waits, with the same
 * bounded mbarrier wait as the GEMM pipeline, on a barrier nothing arrives on.
 * After `limit_ns` (1 ns .. 10 s) the wait gives up and records a timeout, so
 * the next convrot_get_error() returns CONVROT_ERR_TIMEOUT and the context
 * remains usable.  (The GEMM's own waits use a 2 s limit.) */
CONVROT_API int convrot_selftest_wait_timeout(uint64_t limit_ns, convrot_stream_t stream);

/* Test entry for the checked variant's reporting path: launches one thread
 * that evaluates a bounds check with an index one past its extent.  No memory
 * is read or written by it.  In the checked library the next
 * convrot_get_error() returns CONVROT_ERR_BOUNDS (and clears it); the release
 * library compiles its checks away, so there the call returns
 * CONVROT_ERR_UNSUPPORTED and launches nothing. */
CONVROT_API int convrot_selftest_bounds_flag(convrot_stream_t stream);

/* Measurement entry for a roofline denominator: launches a kernel of four
 * 256-thread CTAs per SM whose warps issue only dense int8 MMAs through the
 * legacy warp-level path (mma.sync m16n8k32 s8 x s8 -> s32; tcgen05 has no
 * int8 kind on this GPU), `iters` rounds of 8 independent MMAs per warp.
 * *ops (host pointer) receives the operation count of the launch (2 per
 * multiply-add); time the launch on `stream` to get the rate.  sink: device
 * int32 buffer of at least 4 * (number of SMs) entries, overwritten. */
CONVROT_API int convrot_probe_mma_s8_rate(int iters, int32_t *sink, size_t sink_bytes, double *ops,
                              convrot_stream_t stream);

/* Test entry for the GEMM's own failure path: convrot_gemm_dequant (widened =
 * 0: Wq int8 [N, K], widened inside the GEMM loop) or convrot_gemm_dequant_w16
 * (widened = 1: Wq fp16-held codes [N, K]) with two changes made for the test:
 * every pipeline wait of the GEMM gives up after `limit_ns` (1 ns .. 10 s)
 * instead of 2 s, and the copy that `producer` (0: the activation tiles,
 * 1: the weight tiles) would issue at its iteration `skip_iteration` (counted
 * over the pipeline stages of the tiles a CTA or CTA pair processes, from 0: a
 * stage holds one K block of 64 when widened = 0 and two when widened = 1) is
 * never issued.  The stage it would fill stays empty, so a consumer's bounded
 * wait expires: every
 * role of the CTA then stops, copies and MMAs in flight are drained, the
 * tensor memory is freed and the kernel returns.  The next convrot_get_error()
 * returns CONVROT_ERR_TIMEOUT; y is partly written; the context stays usable.
 * Arguments as in convrot_gemm_dequant (no bias). */
CONVROT_API int convrot_selftest_gemm_fault(int widened, const uint16_t *xq, const float *scale_x, int64_t M,
                                int64_t K, const void *Wq, const float *scale_w, int64_t N, uint16_t *y,
                                uint64_t limit_ns, int64_t skip_iteration, int producer,
                                convrot_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H */
