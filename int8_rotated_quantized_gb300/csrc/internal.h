// Host-side launchers shared between the translation units of libconvrot.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace convrot {

cudaError_t launch_rotq_bf16(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int block,
                             const float *lora_A, const float *lora_B, int rank, float coef, bool out_f16,
                             void *q, float *scale, cudaStream_t st);

// 32-elements-per-thread variants (rotq_wide.cu): usable when the row length
// is a multiple of 32 and pointers/strides allow 32-byte accesses.
bool rotq_wide_ok(const void *x, int64_t K, int64_t ldx, const void *q);
cudaError_t launch_rotq_wide(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int block, bool out_f16, void *q,
                             float *scale, cudaStream_t st);
// Fused LoRA merge + rotate + quantize with rows split along K over a cluster
// (lora_rotq.cu): rank <= 16, K = (2 to 8 CTAs or 1) x a power-of-two slice.
bool lora_cluster_ok(const void *W, int64_t K, int64_t ldw, int block, const float *A, int rank, const void *q);
cudaError_t launch_lora_cluster(const uint16_t *W, int64_t rows, int64_t K, int64_t ldw, int block, const float *A,
                                const float *B, int rank, float coef, int8_t *q, float *scale, unsigned *err,
                                cudaStream_t st);
// The device error word of the current device (convrot_api.cu), or null.
unsigned *current_error_word();
bool lookup_wide_ok(const void *Eq, int64_t D, const void *out);
cudaError_t launch_lookup_wide(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e, int64_t V,
                               int64_t D, int block, uint16_t *out, unsigned *err, cudaStream_t st);


cudaError_t launch_emb_lookup(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e, int64_t V,
                              int64_t D, int block, uint16_t *out, unsigned *err, cudaStream_t st);

// One-off int8 backward weight (bwd_weight.cu); `work` holds
// bwd_weight_work_bytes(N, K) bytes (per-tile column maxima and bounds).
size_t bwd_weight_work_bytes(int64_t N, int64_t K);
cudaError_t launch_bwd_prep_df(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, void *work,
                               int8_t *WtQ, float *scale_wt, cudaStream_t st);

// bf16-mode backward weight (bwd_prep.cu): T [K, N] bf16 = bf16((s_w (.) Wq) R)^T.
// b <= 128 on the tensor cores (bounded waits; a timeout sets DEVERR_TIMEOUT in err).
cudaError_t launch_dequant_t(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, uint16_t *T,
                             unsigned *err, cudaStream_t st);

cudaError_t launch_widen_i8(const int8_t *A, int64_t count, uint16_t *out, cudaStream_t st);

// C[M,N] = A[M,K] . B[N,K]^T with A fp16-held integer codes and B int8 codes.
// out_s32: write the exact int32 accumulator to `out`; otherwise write
// bf16(float(acc) * (sa[m] * sb[n]) + bias[n]).
cudaError_t launch_gemm(const uint16_t *A, const float *sa, const int8_t *B, const float *sb, const uint16_t *bias,
                        int64_t M, int64_t N, int64_t K, void *out, bool out_s32, unsigned *err, cudaStream_t st);

// The dequantization GEMM on weight codes already widened to fp16 values
// (B16 [N, K], from launch_widen_codes): same result as launch_gemm.
cudaError_t launch_gemm_w16(const uint16_t *A, const float *sa, const uint16_t *B16, const float *sb,
                            const uint16_t *bias, int64_t M, int64_t N, int64_t K, uint16_t *out, unsigned *err,
                            cudaStream_t st);
// The same with the LoRA bypass term y += sum_j xa[m, j] lora_b[n, j]: the
// operands divided by the output's scales (xa[m] / dx[m], lora_b[n] / dw[n], d
// = the scale or 1 where it is 0) as three bf16 parts per value
// (kLoraPartsRow = 64 bf16 per row: hi at columns 0-15, mid at 16-31, lo at
// 32-47, zeros at 48-63; j >= rank zero), xa_parts [M][64] and b_parts [N][64]
// from launch_lora_operands.  The GEMM adds the term to each tile's last
// integer chunk as one more K block on the tensor cores.
constexpr int kLoraPartsRow = 64;
cudaError_t launch_gemm_w16_lora(const uint16_t *A, const float *sa, const uint16_t *B16, const float *sb,
                                 const uint16_t *bias, const uint16_t *xa_parts, const uint16_t *b_parts, int64_t M,
                                 int64_t N, int64_t K, uint16_t *out, unsigned *err, cudaStream_t st);
// K spans of the tensor-core down-projection for M rows of length K (lora_down.cu).
int lora_down_spans(int64_t M, int64_t K);
// The bypass operands (lora_down.cu), one cluster kernel: b_parts [N][64] (the
// parts of B[n] / dw[n]) and xa_parts [M][64] = the parts of (coef * x A^T)[m]
// / dx[m], the product computed on the tensor cores.  K % 32 == 0.
cudaError_t launch_lora_operands(const uint16_t *x, const float *scale_x, int64_t M, int64_t K, const float *A,
                                 const float *B, const float *scale_w, int64_t N, int rank, float coef,
                                 uint16_t *xa_parts, uint16_t *b_parts, unsigned *err, cudaStream_t st);
// int8 codes -> fp16 values holding the same integers, 32 per thread (rotq_wide.cu).
cudaError_t launch_widen_codes(const int8_t *A, int64_t count, uint16_t *out, cudaStream_t st);

// P[M,N] = float(A[M,K] . B16[N,K]^T) * sa[m] in fp32 (exact integer sums).
cudaError_t launch_gemm_w16_scale_f32(const uint16_t *A, const float *sa, const uint16_t *B16, int64_t M, int64_t N,
                                      int64_t K, float *out, unsigned *err, cudaStream_t st);
// Second reading of the int8 backward (bwd_r2.cu).
bool bwd_r2_ok(int64_t N, int64_t K, const void *dY, const void *dX);
cudaError_t launch_scaleq(const uint16_t *dY, int64_t M, int64_t N, const float *colscale, uint16_t *q, float *scale,
                          cudaStream_t st);
cudaError_t launch_transpose_widen(const int8_t *W, int64_t N, int64_t K, uint16_t *T, cudaStream_t st);
cudaError_t launch_rot_rows_f32(const float *P, int64_t rows, int64_t L, int block, uint16_t *out, cudaStream_t st);

// C[M,N] = bf16(A[M,K] . B[N,K]^T) with bf16 operands, fp32 accumulation.
cudaError_t launch_gemm_bf16(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K, uint16_t *out,
                             unsigned *err, cudaStream_t st);

// Failure-path self-test of the GEMM itself: the dequantization GEMM (int8
// weight codes widened in the loop, or already widened to fp16 values) with
// every pipeline wait bounded by limit_ns, and the copy of producer `role` at
// its iteration `skip_it` never issued (gemm_tc.cu).
cudaError_t launch_gemm_fault_selftest(bool widened, const uint16_t *A, const float *sa, const void *B,
                                      const float *sb, int64_t M, int64_t N, int64_t K, uint16_t *out, unsigned *err,
                                      uint64_t limit_ns, int skip_it, int role, cudaStream_t st);

// Self-test of the checked build's bounds flag (selftest.cu): false (nothing
// launched) in release builds.
bool launch_bounds_flag_selftest(cudaStream_t st, cudaError_t *e);
// Self-test of the bounded-wait failure path (selftest.cu).
cudaError_t launch_wait_timeout(uint64_t limit_ns, unsigned *err, cudaStream_t st);

}  // namespace convrot
