/*
 * ConvRot INT8 linear layer -- CPU ORACLE (test infrastructure only).
 *
 * This file is the plain, slow, obviously-correct restatement of what the
 * ConvRot INT8 layer computes.  It exists to check the CUDA library; only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources restated (page title, section):
 *   [guide]  "LoRA Training Guide for MOSS-Image" (docs/moss_image_train_network.md),
 *            section 7.1 "VRAM Usage Optimization", paragraph "ConvRot INT8":
 *            block-diagonal Hadamard rotation, per-channel int8 weights,
 *            online activation rotation + dynamic row-wise int8 activation
 *            quantization + dequantization fused into the matmul; the int8
 *            backward option routes grad_x through the same int8 GEMM.
 *   [pr]     sd-scripts pull request #2461 "ConvRot INT8", Summary bullets on
 *            convrot_int8_kernels.py (rotation, row-wise int8, fused GEMM with
 *            dequantization epilogue), convrot_int8_utils.py (frozen base:
 *            grad_x only; fp32 weight_scale; the token embedding quantized in
 *            the rotated basis, so a lookup dequantizes and applies the
 *            inverse rotation).
 *   [forge]  voxprint-model-forge MOSS page, LoRA export: the adapter is merged
 *            as W + scale * (alpha / rank) * B @ A.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes of the repository):
 *   R1  H_b is the Sylvester Hadamard matrix (H_1 = [1], H_2n = [[H,H],[H,-H]]),
 *       normalised by 1/sqrt(b), applied to contiguous blocks of b along the
 *       contraction dimension: R = I (x) H_b / sqrt(b).
 *   R2  Symmetric absmax scale s = max|v| / 127 stored as fp32; codes are
 *       round-half-to-even(v / s) clamped to [-127, 127]; an all-zero row has
 *       s = 0 and codes 0.
 *   R3  The rotation is exact (fp64 here).  The code decision is taken in fp32,
 *       the precision of the GPU kernel: q = rne(fp32(u) * fp32(127 / max|fp32(u)|))
 *       with u the unnormalised block transform H_b x, which equals
 *       rne(v / s) in exact arithmetic.
 *   R4  The dequantization epilogue is y = bf16_rne(acc * s_x * s_w + bias),
 *       evaluated here in fp64.
 *   R5  LoRA merge: W' = bf16_rne(W + c * sum_j B[n,j] A[j,k]), c = fp32(scale*alpha/rank);
 *       the rounding to bf16 decides every later code, so it is taken in fp32
 *       with a sequential fused multiply-add over j, the kernel's precision.
 *   R6  int8 backward: W_eff = (s_w (.) Wq) R (the dequantized base, rotated
 *       back, kept in fp64), WtQ/s_wt = ConvRot quantization of the rows of
 *       W_eff^T along N, dY quantized the same way along N, and
 *       dX = bf16(acc * s_dy * s_wt).
 *   R7  Embedding lookup: out[t] = bf16_rne((s[id] * Eq[id,:]) R), fp64; an id
 *       outside [0, V) yields a zero row and is counted.
 *   R10 int8 backward, second reading: s_w folded into the columns of dY, dY
 *       quantized per row without rotation, the int8 GEMM on Wq as it is
 *       (contraction over N), the rotation along K applied to the product.
 *   R9  LoRA bypass in the forward: instead of merging, the adapter's branch
 *       c * (x A^T) B^T on the unrotated input is added to the dequantized
 *       product before the output rounding (fp64 here).
 *   R8  bf16 backward (the default mode of the pages' backward option): the
 *       frozen base is dequantized transiently, W_eff = bf16_rne((s_w (.) Wq) R)
 *       (fp64 before the rounding), and dX = bf16_rne(dY . W_eff) summed in fp64.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math: the
 * fp32 decisions of R3/R5 rely on IEEE single precision without contraction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 ---- */

/* Exact value of a bf16 bit pattern (the upper 16 bits of an IEEE binary32). */
static double bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in a single rounding. */
static uint16_t f64_to_bf16(double v)
{
    if (v != v)
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int ulp_exp = e - 8;          /* 8 significant bits */
    if (ulp_exp < -133)
        ulp_exp = -133;           /* subnormal spacing 2^-126 * 2^-7 */
    double q = rint(ldexp(a, -ulp_exp));   /* default mode: nearest, ties even */
    double r = ldexp(q, ulp_exp);
    if (r > 0x1.fep127)
        return sign | 0x7f80;
    float f = (float)r;           /* exact: r is representable in bf16 */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

/* ------------------------------------------------------------ Hadamard ---- */

static int is_pow2(int b) { return b >= 1 && (b & (b - 1)) == 0; }

/* Sylvester construction, unnormalised: H_1 = [1]; H_2n = [[H_n, H_n], [H_n, -H_n]]. */
int oracle_hadamard(int b, double *H)
{
    if (!is_pow2(b) || b > 4096)
        return 1;
    H[0] = 1.0;
    for (int n = 1; n < b; n *= 2) {
        for (int i = 0; i < n; i++)
            for (int j = 0; j < n; j++) {
                double h = H[i * b + j];
                H[i * b + (j + n)] = h;
                H[(i + n) * b + j] = h;
                H[(i + n) * b + (j + n)] = -h;
            }
    }
    return 0;
}

/* u = x H_b on every contiguous block of b (unnormalised), explicit O(b^2)
 * matrix-vector products.  H_b is symmetric, so x H_b = (H_b x)^T. */
static void block_transform(const double *H, int b, const double *x, int64_t K, double *u)
{
    for (int64_t k0 = 0; k0 < K; k0 += b)
        for (int j = 0; j < b; j++) {
            double acc = 0.0;
            for (int i = 0; i < b; i++)
                acc += x[k0 + i] * H[i * b + j];
            u[k0 + j] = acc;
        }
}

/* Public for the self-tests: out = x (I (x) H_b / sqrt(b)) row by row, fp64. */
int oracle_rotate_rows(const double *x, int64_t rows, int64_t K, int b, double *out)
{
    if (!is_pow2(b) || K % b != 0)
        return 1;
    double *H = malloc(sizeof(double) * (size_t)b * b);
    if (!H)
        return 2;
    oracle_hadamard(b, H);
    double inv = 1.0 / sqrt((double)b);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        block_transform(H, b, x + r * K, K, out + r * K);
        for (int64_t k = 0; k < K; k++)
            out[r * K + k] *= inv;
    }
    free(H);
    return 0;
}

/* ------------------------------------------------ row-wise quantization ---- */

/* One row: rotate (R1), absmax scale (R2), fp32 code decision (R3). */
static void quantize_row(const double *H, int b, const double *x, int64_t K,
                         double *u, int8_t *q, float *s)
{
    block_transform(H, b, x, K, u);
    double amax = 0.0;
    for (int64_t k = 0; k < K; k++)
        if (fabs(u[k]) > amax)
            amax = fabs(u[k]);
    amax /= sqrt((double)b);                       /* max |v|, v = u / sqrt(b) */
    if (amax == 0.0) {
        *s = 0.0f;
        memset(q, 0, (size_t)K);
        return;
    }
    *s = (float)(amax / 127.0);
    float amax_u = 0.0f;
    for (int64_t k = 0; k < K; k++) {
        float a = fabsf((float)u[k]);
        if (a > amax_u)
            amax_u = a;
    }
    if (amax_u == 0.0f) {
        memset(q, 0, (size_t)K);
        return;
    }
    float inv = 127.0f / amax_u;
    for (int64_t k = 0; k < K; k++) {
        float t = rintf((float)u[k] * inv);
        if (t > 127.0f)
            t = 127.0f;
        if (t < -127.0f)
            t = -127.0f;
        q[k] = (int8_t)t;
    }
}

static int quantize_rows_f64(const double *x, int64_t rows, int64_t K, int64_t ldx, int b,
                             int8_t *q, float *s)
{
    if (!is_pow2(b) || K % b != 0 || rows < 0 || ldx < K)
        return 1;
    double *H = malloc(sizeof(double) * (size_t)b * b);
    if (!H)
        return 2;
    oracle_hadamard(b, H);
    int fail = 0;
#pragma omp parallel
    {
        double *row = malloc(sizeof(double) * (size_t)K);
        double *u = malloc(sizeof(double) * (size_t)K);
        if (!row || !u) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; r++) {
                memcpy(row, x + r * ldx, sizeof(double) * (size_t)K);
                quantize_row(H, b, row, K, u, q + r * K, s + r);
            }
        }
        free(row);
        free(u);
    }
    free(H);
    return fail ? 2 : 0;
}

/* Rotate + quantize rows given in fp64 (R1-R3).  q is [rows, K] contiguous. */
int oracle_quantize_rows_f64(const double *x, int64_t rows, int64_t K, int64_t ldx, int b,
                             int8_t *q, float *s)
{
    return quantize_rows_f64(x, rows, K, ldx, b, q, s);
}

/* Rotate + quantize bf16 rows (weights, activations, embedding table). */
int oracle_quantize_rows_bf16(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, int b,
                              int8_t *q, float *s)
{
    if (!is_pow2(b) || K % b != 0 || rows < 0 || ldx < K)
        return 1;
    double *H = malloc(sizeof(double) * (size_t)b * b);
    if (!H)
        return 2;
    oracle_hadamard(b, H);
    int fail = 0;
#pragma omp parallel
    {
        double *row = malloc(sizeof(double) * (size_t)K);
        double *u = malloc(sizeof(double) * (size_t)K);
        if (!row || !u) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; r++) {
                for (int64_t k = 0; k < K; k++)
                    row[k] = bf16_to_f64(x[r * ldx + k]);
                quantize_row(H, b, row, K, u, q + r * K, s + r);
            }
        }
        free(row);
        free(u);
    }
    free(H);
    return fail ? 2 : 0;
}

/* ------------------------------------------------------------ LoRA (R5) ---- */

/* Merge W' = bf16(W + c * B@A), c = fp32(scale * alpha / rank); A fp32 [r, K],
 * B fp32 [N, r].  Out is [N, K] contiguous bf16 bits. */
int oracle_lora_merge(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                      const float *A, const float *B, int rank, float alpha, float scale,
                      uint16_t *out)
{
    if (rank <= 0 || ldw < K)
        return 1;
    float c = (float)((double)scale * (double)alpha / (double)rank);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            float d = 0.0f;
            for (int j = 0; j < rank; j++)
                d = fmaf(B[n * rank + j], A[(int64_t)j * K + k], d);
            float w = (float)bf16_to_f64(W[n * ldw + k]);
            out[n * K + k] = f64_to_bf16((double)fmaf(c, d, w));
        }
    return 0;
}

/* Weight quantization at load (merge first when A and B are given, then quantize). */
int oracle_quantize_weight(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int b,
                           const float *A, const float *B, int rank, float alpha, float scale,
                           int8_t *Wq, float *s_w)
{
    if (A == NULL || B == NULL)
        return oracle_quantize_rows_bf16(W, N, K, ldw, b, Wq, s_w);
    uint16_t *m = malloc(sizeof(uint16_t) * (size_t)N * (size_t)K);
    if (!m)
        return 2;
    int rc = oracle_lora_merge(W, N, K, ldw, A, B, rank, alpha, scale, m);
    if (rc == 0)
        rc = oracle_quantize_rows_bf16(m, N, K, K, b, Wq, s_w);
    free(m);
    return rc;
}

/* ----------------------------------------------------------- GEMM (int) ---- */

/* C[m,n] = sum_k A[m,k] B[n,k], accumulated in int64; returns 3 if a result
 * does not fit in int32. */
int oracle_gemm_s32(const int8_t *A, const int8_t *B, int64_t M, int64_t N, int64_t K, int32_t *C)
{
    int overflow = 0;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; k++)
                acc += (int64_t)A[m * K + k] * (int64_t)B[n * K + k];
            if (acc > INT32_MAX || acc < INT32_MIN) {
#pragma omp atomic write
                overflow = 1;
            }
            C[m * N + n] = (int32_t)acc;
        }
    return overflow ? 3 : 0;
}

/* Dequantization epilogue (R4): y = bf16(acc * s_a[m] * s_b[n] + bias[n]) in fp64. */
int oracle_dequant(const int32_t *acc, int64_t M, int64_t N, const float *s_a, const float *s_b,
                   const uint16_t *bias, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double v = (double)acc[m * N + n] * (double)s_a[m] * (double)s_b[n];
            if (bias)
                v += bf16_to_f64(bias[n]);
            y[m * N + n] = f64_to_bf16(v);
        }
    return 0;
}

/* ------------------------------------------------------ linear forward ---- */

/* y = dequant(quant(x R) . Wq^T).  xq/s_x receive the activation codes when non-null. */
int oracle_linear_fwd(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq, const float *s_w,
                      int64_t N, int b, const uint16_t *bias, uint16_t *y,
                      int8_t *xq_out, float *sx_out)
{
    int8_t *xq = xq_out ? xq_out : malloc((size_t)M * (size_t)K);
    float *sx = sx_out ? sx_out : malloc(sizeof(float) * (size_t)M);
    int32_t *acc = malloc(sizeof(int32_t) * (size_t)M * (size_t)N);
    int rc = 2;
    if (xq && sx && acc) {
        rc = oracle_quantize_rows_bf16(x, M, K, K, b, xq, sx);
        if (rc == 0)
            rc = oracle_gemm_s32(xq, Wq, M, N, K, acc);
        if (rc == 0)
            rc = oracle_dequant(acc, M, N, sx, s_w, bias, y);
    }
    if (!xq_out)
        free(xq);
    if (!sx_out)
        free(sx);
    free(acc);
    return rc;
}

/* LoRA bypass in the forward (R9): the adapter is not merged into W; its
 * branch sees the unrotated input and is added before the output rounding:
 *   y = bf16(acc * s_x * s_w + bias + c * sum_j (sum_k x[m,k] A[j,k]) B[n,j])
 * in fp64, c = fp32(scale * alpha / rank), A [rank, K], B [N, rank] fp32. */
int oracle_linear_fwd_lora(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq, const float *s_w,
                           int64_t N, int b, const uint16_t *bias, const float *A, const float *B, int rank,
                           float alpha, float scale, uint16_t *y)
{
    if (rank <= 0)
        return 1;
    int8_t *xq = malloc((size_t)M * (size_t)K);
    float *sx = malloc(sizeof(float) * (size_t)M);
    int32_t *acc = malloc(sizeof(int32_t) * (size_t)M * (size_t)N);
    double *xa = malloc(sizeof(double) * (size_t)M * (size_t)rank);
    int rc = 2;
    if (xq && sx && acc && xa) {
        rc = oracle_quantize_rows_bf16(x, M, K, K, b, xq, sx);
        if (rc == 0)
            rc = oracle_gemm_s32(xq, Wq, M, N, K, acc);
        if (rc == 0) {
            double c = (double)(float)((double)scale * (double)alpha / (double)rank);
#pragma omp parallel for schedule(static)
            for (int64_t m = 0; m < M; m++)
                for (int j = 0; j < rank; j++) {
                    double d = 0.0;
                    for (int64_t k = 0; k < K; k++)
                        d += bf16_to_f64(x[m * K + k]) * (double)A[(int64_t)j * K + k];
                    xa[m * rank + j] = d;
                }
#pragma omp parallel for schedule(static)
            for (int64_t m = 0; m < M; m++)
                for (int64_t n = 0; n < N; n++) {
                    double v = (double)acc[m * N + n] * (double)sx[m] * (double)s_w[n];
                    if (bias)
                        v += bf16_to_f64(bias[n]);
                    double l = 0.0;
                    for (int j = 0; j < rank; j++)
                        l += xa[m * rank + j] * (double)B[n * rank + j];
                    y[m * N + n] = f64_to_bf16(v + c * l);
                }
        }
    }
    free(xq);
    free(sx);
    free(acc);
    free(xa);
    return rc;
}

/* ---------------------------------------------------- int8 backward (R6) ---- */

/* W_eff = (s_w (.) Wq) R along K in fp64; WtQ/s_wt = quantization of the rows
 * of W_eff^T ([K, N]) along N.  WtQ is [K, N] int8, s_wt is [K]. */
int oracle_prepare_bwd_weight(const int8_t *Wq, const float *s_w, int64_t N, int64_t K, int b,
                              int8_t *WtQ, float *s_wt)
{
    if (!is_pow2(b) || K % b != 0 || N % b != 0)
        return 1;
    double *deq = malloc(sizeof(double) * (size_t)N * (size_t)K);
    double *eff = malloc(sizeof(double) * (size_t)N * (size_t)K);
    double *effT = malloc(sizeof(double) * (size_t)N * (size_t)K);
    int rc = 2;
    if (deq && eff && effT) {
        for (int64_t n = 0; n < N; n++)
            for (int64_t k = 0; k < K; k++)
                deq[n * K + k] = (double)s_w[n] * (double)Wq[n * K + k];
        rc = oracle_rotate_rows(deq, N, K, b, eff);
        if (rc == 0) {
            for (int64_t n = 0; n < N; n++)
                for (int64_t k = 0; k < K; k++)
                    effT[k * N + n] = eff[n * K + k];
            rc = quantize_rows_f64(effT, K, N, N, b, WtQ, s_wt);
        }
    }
    free(deq);
    free(eff);
    free(effT);
    return rc;
}

/* dX = dequant(quant(dY R_N) . WtQ^T): dY [M, N] bf16, WtQ [K, N], dX [M, K]. */
int oracle_linear_bwd_x(const uint16_t *dY, int64_t M, int64_t N, const int8_t *WtQ,
                        const float *s_wt, int64_t K, int b, uint16_t *dX,
                        int8_t *dyq_out, float *sdy_out)
{
    return oracle_linear_fwd(dY, M, N, WtQ, s_wt, K, b, NULL, dX, dyq_out, sdy_out);
}

/* ---------------------------------------------- bf16 backward (R8) ---- */

/* The default backward mode of the pages: the frozen base is dequantized
 * transiently and grad_x is a bf16 matmul.  W_eff = bf16((s_w (.) Wq) R) along
 * K, written transposed: WeffT [K, N] bf16 bits. */
int oracle_dequant_weight_t(const int8_t *Wq, const float *s_w, int64_t N, int64_t K, int b, uint16_t *WeffT)
{
    if (!is_pow2(b) || K % b != 0)
        return 1;
    double *deq = malloc(sizeof(double) * (size_t)N * (size_t)K);
    double *eff = malloc(sizeof(double) * (size_t)N * (size_t)K);
    int rc = 2;
    if (deq && eff) {
        for (int64_t n = 0; n < N; n++)
            for (int64_t k = 0; k < K; k++)
                deq[n * K + k] = (double)s_w[n] * (double)Wq[n * K + k];
        rc = oracle_rotate_rows(deq, N, K, b, eff);
        if (rc == 0)
            for (int64_t n = 0; n < N; n++)
                for (int64_t k = 0; k < K; k++)
                    WeffT[k * N + n] = f64_to_bf16(eff[n * K + k]);
    }
    free(deq);
    free(eff);
    return rc;
}

/* C[m, n] = bf16(sum_k A[m, k] B[n, k]) with bf16 inputs, summed in fp64. */
int oracle_gemm_bf16(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K, uint16_t *C)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++)
                acc += bf16_to_f64(A[m * K + k]) * bf16_to_f64(B[n * K + k]);
            C[m * N + n] = f64_to_bf16(acc);
        }
    return 0;
}

/* ----------------------------------- int8 backward, second reading (R10) ---- */

/* The scale of the frozen weight is folded into the columns of dY, which is
 * quantized per row without a rotation, and the int8 GEMM takes Wq as it is
 * (contraction over N); the rotation along K is applied to the product:
 *   D   = fp32(dY[m,n] * s_w[n]),  Dq, s_d = per-row absmax codes of D
 *   dX  = bf16( (s_d[m] * sum_n Dq[m,n] Wq[n,k]) R )   (fp64 here). */
int oracle_linear_bwd_x_r2(const uint16_t *dY, int64_t M, int64_t N, const int8_t *Wq, const float *s_w,
                           int64_t K, int b, uint16_t *dX, int8_t *dq_out, float *sd_out)
{
    if (!is_pow2(b) || K % b != 0)
        return 1;
    double *D = malloc(sizeof(double) * (size_t)M * (size_t)N);
    int8_t *dq = dq_out ? dq_out : malloc((size_t)M * (size_t)N);
    float *sd = sd_out ? sd_out : malloc(sizeof(float) * (size_t)M);
    int8_t *wt = malloc((size_t)N * (size_t)K);
    int32_t *acc = malloc(sizeof(int32_t) * (size_t)M * (size_t)K);
    double *v = malloc(sizeof(double) * (size_t)M * (size_t)K);
    double *vr = malloc(sizeof(double) * (size_t)M * (size_t)K);
    int rc = 2;
    if (D && dq && sd && wt && acc && v && vr) {
        for (int64_t m = 0; m < M; m++)
            for (int64_t n = 0; n < N; n++)
                D[m * N + n] = (double)((float)bf16_to_f64(dY[m * N + n]) * s_w[n]);
        rc = quantize_rows_f64(D, M, N, N, 1, dq, sd);
        if (rc == 0) {
            for (int64_t n = 0; n < N; n++)
                for (int64_t k = 0; k < K; k++)
                    wt[k * N + n] = Wq[n * K + k];
            rc = oracle_gemm_s32(dq, wt, M, K, N, acc);
        }
        if (rc == 0) {
            for (int64_t m = 0; m < M; m++)
                for (int64_t k = 0; k < K; k++)
                    v[m * K + k] = (double)sd[m] * (double)acc[m * K + k];
            rc = oracle_rotate_rows(v, M, K, b, vr);
        }
        if (rc == 0)
            for (int64_t i = 0; i < M * K; i++)
                dX[i] = f64_to_bf16(vr[i]);
    }
    free(D);
    if (!dq_out)
        free(dq);
    if (!sd_out)
        free(sd);
    free(wt);
    free(acc);
    free(v);
    free(vr);
    return rc;
}

/* ------------------------------------------------- embedding lookup (R7) ---- */

int oracle_embedding_lookup(const int64_t *ids, int64_t n, const int8_t *Eq, const float *s_e,
                            int64_t V, int64_t D, int b, uint16_t *out, int64_t *bad)
{
    if (!is_pow2(b) || D % b != 0)
        return 1;
    double *H = malloc(sizeof(double) * (size_t)b * b);
    if (!H)
        return 2;
    oracle_hadamard(b, H);
    double inv = 1.0 / sqrt((double)b);
    int64_t nbad = 0;
#pragma omp parallel reduction(+ : nbad)
    {
        double *row = malloc(sizeof(double) * (size_t)D);
        double *u = malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; t++) {
            int64_t id = ids[t];
            if (id < 0 || id >= V) {
                nbad++;
                for (int64_t d = 0; d < D; d++)
                    out[t * D + d] = 0;
                continue;
            }
            for (int64_t d = 0; d < D; d++)
                row[d] = (double)s_e[id] * (double)Eq[id * D + d];
            block_transform(H, b, row, D, u);
            for (int64_t d = 0; d < D; d++)
                out[t * D + d] = f64_to_bf16(u[d] * inv);
        }
        free(row);
        free(u);
    }
    free(H);
    if (bad)
        *bad = nbad;
    return 0;
}

/* -------------------------------------------------------------- misc ---- */

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* bf16 helpers exported for the self-tests (they pin the conversions). */
double oracle_bf16_to_f64(uint16_t h) { return bf16_to_f64(h); }
uint16_t oracle_f64_to_bf16(double v) { return f64_to_bf16(v); }
