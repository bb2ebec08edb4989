// C ABI of libconvrot: argument validation, workspace carving and dispatch to
// the kernels.  Every entry point checks its arguments on the host and returns
// a status before enqueuing anything; kernels report device-side conditions
// through one sticky error word per device (read by convrot_get_error).
#include <math.h>

#include <mutex>

#include "convrot.h"
#include "common.cuh"
#include "internal.h"

namespace {

__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices] = {nullptr};
int g_cc_ok[kMaxDevices] = {0};  // 0 unknown, 1 supported, -1 unsupported
std::mutex g_mu;

// Per-device set-up: the device address of the error word and whether the
// device can run the sm_103a code in this library.
int device_setup(unsigned **err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CONVROT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_cc_ok[dev] == 1) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
                g_cc_ok[dev] = 0;
                return CONVROT_ERR_CUDA;
            }
            g_err_ptr[dev] = static_cast<unsigned *>(p);
        }
    }
    if (g_cc_ok[dev] != 1) return CONVROT_ERR_UNSUPPORTED;
    *err = g_err_ptr[dev];
    return CONVROT_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool block_ok(int b) { return b == 8 || b == 16 || b == 32 || b == 64 || b == 128 || b == 256; }
// Longest contraction of the integer GEMM entry points: 127 * 127 * 2^17 < 2^31, so the int32 accumulator
// cannot overflow for any codes in [-127, 127].
constexpr int64_t kMaxIntK = int64_t(1) << 17;
bool row_ok(int64_t K, int b) { return K > 0 && K % b == 0 && K % 16 == 0 && K <= CONVROT_MAX_ROW; }
size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA; }

#ifdef CONVROT_CHECKED
// The bounds flags of the checked build, one per translation unit.
std::mutex &bounds_mu() {
    static std::mutex mu;
    return mu;
}
unsigned (*g_bounds_readers[32])() = {nullptr};
int g_bounds_count = 0;
#endif

#define CHECK(cond)                                   \
    do {                                              \
        if (!(cond)) return CONVROT_ERR_INVALID_ARG; \
    } while (0)

int quantize_act_impl(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int block, uint16_t *xq, float *sx,
                      cudaStream_t st) {
    return cuda_status(convrot::launch_rotq_bf16(x, M, K, ldx, block, nullptr, nullptr, 0, 0.f, true, xq, sx, st));
}

int gemm_impl(const uint16_t *xq, const float *sx, int64_t M, int64_t K, const int8_t *Wq, const float *sw, int64_t N,
              const uint16_t *bias, uint16_t *y, unsigned *err, cudaStream_t st) {
    return cuda_status(convrot::launch_gemm(xq, sx, Wq, sw, bias, M, N, K, y, false, err, st));
}

}  // namespace

namespace convrot {
#ifdef CONVROT_CHECKED
void register_bounds_flag(unsigned (*read_and_clear)()) {
    std::lock_guard<std::mutex> lock(bounds_mu());
    if (g_bounds_count < 32) g_bounds_readers[g_bounds_count++] = read_and_clear;
}
#endif
unsigned *current_error_word() {
    unsigned *err = nullptr;
    return device_setup(&err) == CONVROT_OK ? err : nullptr;
}
}  // namespace convrot

extern "C" {

const char *convrot_status_string(int status) {
    switch (status) {
        case CONVROT_OK: return "CONVROT_OK";
        case CONVROT_ERR_INVALID_ARG: return "CONVROT_ERR_INVALID_ARG";
        case CONVROT_ERR_UNSUPPORTED: return "CONVROT_ERR_UNSUPPORTED";
        case CONVROT_ERR_CUDA: return "CONVROT_ERR_CUDA";
        case CONVROT_ERR_TIMEOUT: return "CONVROT_ERR_TIMEOUT";
        case CONVROT_ERR_INDEX: return "CONVROT_ERR_INDEX";
        case CONVROT_ERR_BOUNDS: return "CONVROT_ERR_BOUNDS";
        default: return "CONVROT_ERR_UNKNOWN";
    }
}

int convrot_version(void) { return 100; }

int convrot_get_error(convrot_stream_t stream) {
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CONVROT_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return CONVROT_ERR_CUDA;
    if (v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return CONVROT_ERR_CUDA;
    }
#ifdef CONVROT_CHECKED
    unsigned bounds = 0u;
    {
        std::lock_guard<std::mutex> lock(bounds_mu());
        for (int i = 0; i < g_bounds_count; ++i) bounds |= g_bounds_readers[i]();
    }
    if (bounds != 0u) return CONVROT_ERR_BOUNDS;
#endif
    if (v & convrot::DEVERR_TIMEOUT) return CONVROT_ERR_TIMEOUT;
    if (v & convrot::DEVERR_INDEX) return CONVROT_ERR_INDEX;
    return CONVROT_OK;
}

int convrot_quantize_weight(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int block, const float *lora_A,
                            const float *lora_B, int rank, float alpha, float scale, int8_t *Wq, float *scale_w,
                            convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && N >= 0 && ldw >= K && ldw % 8 == 0);
    CHECK(N == 0 || (W && Wq && scale_w && aligned16(W) && aligned16(Wq)));
    CHECK((lora_A == nullptr) == (lora_B == nullptr));
    if (lora_A) CHECK(rank >= 1 && rank <= 64 && aligned16(lora_A) && ((uintptr_t)lora_B & 3u) == 0);
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (N == 0) return CONVROT_OK;
    const float coef = lora_A ? (float)((double)scale * (double)alpha / (double)rank) : 0.f;
    if (lora_A && convrot::lora_cluster_ok(W, K, ldw, block, lora_A, rank, Wq))
        return cuda_status(convrot::launch_lora_cluster(W, N, K, ldw, block, lora_A, lora_B, rank, coef, Wq, scale_w,
                                                        err, (cudaStream_t)stream));
    return cuda_status(convrot::launch_rotq_bf16(W, N, K, ldw, block, lora_A, lora_B, lora_A ? rank : 0, coef, false,
                                                 Wq, scale_w, (cudaStream_t)stream));
}

int convrot_quantize_activation(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int block, uint16_t *xq,
                                float *scale_x, convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && M >= 0 && ldx >= K && ldx % 8 == 0);
    CHECK(M == 0 || (x && xq && scale_x && aligned16(x) && aligned16(xq)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0) return CONVROT_OK;
    return quantize_act_impl(x, M, K, ldx, block, xq, scale_x, (cudaStream_t)stream);
}

int convrot_gemm_dequant(const uint16_t *xq, const float *scale_x, int64_t M, int64_t K, const int8_t *Wq,
                         const float *scale_w, int64_t N, const uint16_t *bias, uint16_t *y,
                         convrot_stream_t stream) {
    CHECK(M >= 0 && N >= 0 && K > 0 && K % 16 == 0 && K <= kMaxIntK && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (xq && scale_x && Wq && scale_w && y && aligned16(xq) && aligned16(Wq) && aligned16(y) &&
           aligned16(scale_x) && aligned16(scale_w) && (bias == nullptr || aligned16(bias))));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    return gemm_impl(xq, scale_x, M, K, Wq, scale_w, N, bias, y, err, (cudaStream_t)stream);
}

size_t convrot_act_workspace_bytes(int64_t M, int64_t K) {
    if (M < 0 || K < 0) return 0;
    return align256((size_t)M * (size_t)K * 2) + align256((size_t)M * 4);
}

size_t convrot_linear_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (M < 0 || K < 0 || N < 0) return 0;
    return convrot_act_workspace_bytes(M, K) + align256((size_t)N * (size_t)K * 2);
}

int convrot_widen_codes(const int8_t *q, int64_t count, uint16_t *out16, convrot_stream_t stream) {
    CHECK(count >= 0 && count % 16 == 0);
    CHECK(count == 0 || (q && out16 && aligned16(q) && aligned16(out16)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (count == 0) return CONVROT_OK;
    return cuda_status(convrot::launch_widen_codes(q, count, out16, (cudaStream_t)stream));
}

int convrot_gemm_dequant_w16(const uint16_t *xq, const float *scale_x, int64_t M, int64_t K, const uint16_t *Wq16,
                             const float *scale_w, int64_t N, const uint16_t *bias, uint16_t *y,
                             convrot_stream_t stream) {
    CHECK(M >= 0 && N >= 0 && K > 0 && K % 16 == 0 && K <= kMaxIntK && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (xq && scale_x && Wq16 && scale_w && y && aligned16(xq) && aligned16(Wq16) && aligned16(y) &&
           aligned16(scale_x) && aligned16(scale_w) && (bias == nullptr || aligned16(bias))));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    return cuda_status(
        convrot::launch_gemm_w16(xq, scale_x, Wq16, scale_w, bias, M, N, K, y, err, (cudaStream_t)stream));
}

int convrot_linear_fwd(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq, const float *scale_w, int64_t N,
                       int block, const uint16_t *bias, uint16_t *y, void *workspace, size_t ws_bytes,
                       convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && M >= 0 && N >= 0 && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (x && Wq && scale_w && y && workspace && aligned16(x) && aligned16(Wq) && aligned16(y) &&
           aligned16(scale_w) && ((uintptr_t)workspace & 255u) == 0 && (bias == nullptr || aligned16(bias))));
    CHECK(M == 0 || N == 0 || ws_bytes >= convrot_act_workspace_bytes(M, K));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint16_t *xq = static_cast<uint16_t *>(workspace);
    float *sx = reinterpret_cast<float *>(static_cast<char *>(workspace) + align256((size_t)M * (size_t)K * 2));
    rc = quantize_act_impl(x, M, K, K, block, xq, sx, st);
    if (rc != CONVROT_OK) return rc;
    if (ws_bytes >= convrot_linear_workspace_bytes(M, K, N)) {
        // transient fp16 copy of the weight codes, then the GEMM without widening in its loop
        uint16_t *w16 = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) + convrot_act_workspace_bytes(M, K));
        rc = cuda_status(convrot::launch_widen_codes(Wq, N * K, w16, st));
        if (rc != CONVROT_OK) return rc;
        return cuda_status(convrot::launch_gemm_w16(xq, sx, w16, scale_w, bias, M, N, K, y, err, st));
    }
    return gemm_impl(xq, sx, M, K, Wq, scale_w, N, bias, y, err, st);
}

size_t convrot_linear_lora_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (M < 0 || K < 0 || N < 0) return 0;
    const size_t parts_row = (size_t)convrot::kLoraPartsRow * 2;
    return convrot_linear_workspace_bytes(M, K, N) + align256((size_t)M * parts_row) + align256((size_t)N * parts_row);
}

int convrot_linear_fwd_lora(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq, const float *scale_w,
                            int64_t N, int block, const uint16_t *bias, const float *lora_A, const float *lora_B,
                            int rank, float alpha, float scale, uint16_t *y, void *workspace, size_t ws_bytes,
                            convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && K % 32 == 0 && M >= 0 && N >= 0 && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX && rank >= 1 && rank <= 16);
    CHECK(M == 0 || N == 0 ||
          (x && Wq && scale_w && y && lora_A && lora_B && workspace && aligned16(x) && aligned16(Wq) &&
           aligned16(y) && aligned16(scale_w) && aligned16(lora_A) && ((uintptr_t)lora_B & 3u) == 0 &&
           ((uintptr_t)workspace & 255u) == 0 && (bias == nullptr || aligned16(bias))));
    CHECK(M == 0 || N == 0 || ws_bytes >= convrot_linear_lora_workspace_bytes(M, K, N));
    const float coef = (float)((double)scale * (double)alpha / (double)rank);
    if (coef == 0.f)  // the branch is zero: the plain forward (its widened-weight path, bit-identical)
        return convrot_linear_fwd(x, M, K, Wq, scale_w, N, block, bias, y, workspace, ws_bytes, stream);
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    uint16_t *xq = reinterpret_cast<uint16_t *>(ws);
    float *sx = reinterpret_cast<float *>(ws + align256((size_t)M * (size_t)K * 2));
    uint16_t *w16 = reinterpret_cast<uint16_t *>(ws + convrot_act_workspace_bytes(M, K));
    const size_t parts_row = (size_t)convrot::kLoraPartsRow * 2;
    char *lw = ws + convrot_linear_workspace_bytes(M, K, N);
    uint16_t *xa_parts = reinterpret_cast<uint16_t *>(lw);
    uint16_t *b_parts = reinterpret_cast<uint16_t *>(lw + align256((size_t)M * parts_row));
    rc = quantize_act_impl(x, M, K, K, block, xq, sx, st);
    if (rc != CONVROT_OK) return rc;
    rc = cuda_status(
        convrot::launch_lora_operands(x, sx, M, K, lora_A, lora_B, scale_w, N, rank, coef, xa_parts, b_parts, err, st));
    if (rc != CONVROT_OK) return rc;
    rc = cuda_status(convrot::launch_widen_codes(Wq, N * K, w16, st));
    if (rc != CONVROT_OK) return rc;
    return cuda_status(
        convrot::launch_gemm_w16_lora(xq, sx, w16, scale_w, bias, xa_parts, b_parts, M, N, K, y, err, st));
}

size_t convrot_bwd_weight_workspace_bytes(int64_t N, int64_t K) {
    if (N < 0 || K < 0) return 0;
    return align256(convrot::bwd_weight_work_bytes(N, K));
}

int convrot_prepare_bwd_weight(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block, int8_t *WtQ,
                               float *scale_wt, void *workspace, size_t ws_bytes, convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && row_ok(N, block));
    CHECK(Wq && scale_w && WtQ && scale_wt && workspace && aligned16(Wq) && aligned16(WtQ) &&
          ((uintptr_t)workspace & 255u) == 0);
    CHECK(ws_bytes >= convrot_bwd_weight_workspace_bytes(N, K));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    return cuda_status(
        convrot::launch_bwd_prep_df(Wq, scale_w, N, K, block, workspace, WtQ, scale_wt, (cudaStream_t)stream));
}

int convrot_linear_bwd_x(const uint16_t *dY, int64_t M, int64_t N, const int8_t *WtQ, const float *scale_wt,
                         int64_t K, int block, uint16_t *dX, void *workspace, size_t ws_bytes,
                         convrot_stream_t stream) {
    // The backward is the forward GEMM with the roles of N and K exchanged.
    return convrot_linear_fwd(dY, M, N, WtQ, scale_wt, K, block, nullptr, dX, workspace, ws_bytes, stream);
}

size_t convrot_bwd_x_r2_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    return convrot_act_workspace_bytes(M, N) + align256((size_t)K * (size_t)N * 2) +
           align256((size_t)M * (size_t)K * sizeof(float));
}

int convrot_linear_bwd_x_r2(const uint16_t *dY, int64_t M, int64_t N, const int8_t *Wq, const float *scale_w,
                            int64_t K, int block, uint16_t *dX, void *workspace, size_t ws_bytes,
                            convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && row_ok(N, 16) && M >= 0 && M <= INT32_MAX);
    CHECK(M == 0 || (dY && Wq && scale_w && dX && workspace && aligned16(Wq) && aligned16(scale_w) &&
                     ((uintptr_t)workspace & 255u) == 0 && convrot::bwd_r2_ok(N, K, dY, dX)));
    CHECK(M == 0 || ws_bytes >= convrot_bwd_x_r2_workspace_bytes(M, N, K));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0) return CONVROT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    uint16_t *dq = reinterpret_cast<uint16_t *>(ws);
    float *sd = reinterpret_cast<float *>(ws + align256((size_t)M * (size_t)N * 2));
    uint16_t *wt16 = reinterpret_cast<uint16_t *>(ws + convrot_act_workspace_bytes(M, N));
    float *P = reinterpret_cast<float *>(ws + convrot_act_workspace_bytes(M, N) + align256((size_t)K * (size_t)N * 2));
    rc = cuda_status(convrot::launch_scaleq(dY, M, N, scale_w, dq, sd, st));
    if (rc != CONVROT_OK) return rc;
    rc = cuda_status(convrot::launch_transpose_widen(Wq, N, K, wt16, st));
    if (rc != CONVROT_OK) return rc;
    // P [M, K] = float(Dq [M, N] . (Wt16 [K, N])^T) * s_d
    rc = cuda_status(convrot::launch_gemm_w16_scale_f32(dq, sd, wt16, M, K, N, P, err, st));
    if (rc != CONVROT_OK) return rc;
    return cuda_status(convrot::launch_rot_rows_f32(P, M, K, block, dX, st));
}

int convrot_dequant_weight_t(const int8_t *Wq, const float *scale_w, int64_t N, int64_t K, int block,
                             uint16_t *WeffT, convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && N >= 0 && N % 16 == 0 && N <= INT32_MAX);
    CHECK(N == 0 || (Wq && scale_w && WeffT && aligned16(Wq) && aligned16(WeffT)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (N == 0) return CONVROT_OK;
    return cuda_status(convrot::launch_dequant_t(Wq, scale_w, N, K, block, WeffT, err, (cudaStream_t)stream));
}

int convrot_gemm_bf16(const uint16_t *A, int64_t M, int64_t K, const uint16_t *B, int64_t N, uint16_t *C,
                      convrot_stream_t stream) {
    CHECK(M >= 0 && N >= 0 && K > 0 && K % 16 == 0 && K <= (1 << 20) && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 || (A && B && C && aligned16(A) && aligned16(B) && aligned16(C)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    return cuda_status(convrot::launch_gemm_bf16(A, B, M, N, K, C, err, (cudaStream_t)stream));
}

size_t convrot_bwd_x_bf16_workspace_bytes(int64_t N, int64_t K) {
    if (N < 0 || K < 0) return 0;
    return align256((size_t)N * (size_t)K * 2);
}

int convrot_linear_bwd_x_bf16(const uint16_t *dY, int64_t M, int64_t N, const int8_t *Wq, const float *scale_w,
                              int64_t K, int block, uint16_t *dX, void *workspace, size_t ws_bytes,
                              convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(K, block) && M >= 0 && N >= 0 && N % 16 == 0 && N <= (1 << 20));
    CHECK(M <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (dY && Wq && scale_w && dX && workspace && aligned16(dY) && aligned16(Wq) && aligned16(dX) &&
           ((uintptr_t)workspace & 255u) == 0 && ws_bytes >= convrot_bwd_x_bf16_workspace_bytes(N, K)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint16_t *weff_t = static_cast<uint16_t *>(workspace);
    rc = cuda_status(convrot::launch_dequant_t(Wq, scale_w, N, K, block, weff_t, err, st));
    if (rc != CONVROT_OK) return rc;
    // dX [M, K] = dY [M, N] . (WeffT [K, N])^T
    return cuda_status(convrot::launch_gemm_bf16(dY, weff_t, M, K, N, dX, err, st));
}

int convrot_embedding_lookup(const int64_t *ids, int64_t n, const int8_t *Eq, const float *scale_e, int64_t V,
                             int64_t D, int block, uint16_t *out, convrot_stream_t stream) {
    CHECK(block_ok(block) && row_ok(D, block) && n >= 0 && V >= 0);
    CHECK(n == 0 || (ids && Eq && scale_e && out && aligned16(Eq) && aligned16(out) && ((uintptr_t)ids & 7u) == 0));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (n == 0) return CONVROT_OK;
    return cuda_status(convrot::launch_emb_lookup(ids, n, Eq, scale_e, V, D, block, out, err, (cudaStream_t)stream));
}

size_t convrot_gemm_s32_workspace_bytes(int64_t M, int64_t K) {
    if (M < 0 || K < 0) return 0;
    return align256((size_t)M * (size_t)K * 2);
}

int convrot_gemm_s32(const int8_t *A, const int8_t *B, int64_t M, int64_t N, int64_t K, int32_t *C, void *workspace,
                     size_t ws_bytes, convrot_stream_t stream) {
    CHECK(M >= 0 && N >= 0 && K > 0 && K % 16 == 0 && K <= kMaxIntK && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (A && B && C && workspace && aligned16(A) && aligned16(B) && aligned16(C) &&
           ((uintptr_t)workspace & 255u) == 0 && ws_bytes >= convrot_gemm_s32_workspace_bytes(M, K)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint16_t *a16 = static_cast<uint16_t *>(workspace);
    rc = cuda_status(convrot::launch_widen_i8(A, M * K, a16, st));
    if (rc != CONVROT_OK) return rc;
    return cuda_status(convrot::launch_gemm(a16, nullptr, B, nullptr, nullptr, M, N, K, C, true, err, st));
}

int convrot_selftest_gemm_fault(int widened, const uint16_t *xq, const float *scale_x, int64_t M, int64_t K,
                                const void *Wq, const float *scale_w, int64_t N, uint16_t *y, uint64_t limit_ns,
                                int64_t skip_iteration, int producer, convrot_stream_t stream) {
    CHECK(limit_ns > 0 && limit_ns <= 10000000000ull && (producer == 0 || producer == 1));
    CHECK(skip_iteration >= 0 && skip_iteration <= INT32_MAX && (widened == 0 || widened == 1));
    CHECK(M >= 0 && N >= 0 && K > 0 && K % 16 == 0 && K <= kMaxIntK && N % 16 == 0);
    CHECK(M <= INT32_MAX && N <= INT32_MAX);
    CHECK(M == 0 || N == 0 ||
          (xq && scale_x && Wq && scale_w && y && aligned16(xq) && aligned16(Wq) && aligned16(y) &&
           aligned16(scale_x) && aligned16(scale_w)));
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    if (M == 0 || N == 0) return CONVROT_OK;
    return cuda_status(convrot::launch_gemm_fault_selftest(widened != 0, xq, scale_x, Wq, scale_w, M, N, K, y, err,
                                                           limit_ns, (int)skip_iteration, producer,
                                                           (cudaStream_t)stream));
}

int convrot_selftest_wait_timeout(uint64_t limit_ns, convrot_stream_t stream) {
    CHECK(limit_ns > 0 && limit_ns <= 10000000000ull);
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    return cuda_status(convrot::launch_wait_timeout(limit_ns, err, (cudaStream_t)stream));
}

int convrot_selftest_bounds_flag(convrot_stream_t stream) {
    unsigned *err = nullptr;
    int rc = device_setup(&err);
    if (rc != CONVROT_OK) return rc;
    cudaError_t e;
    if (!convrot::launch_bounds_flag_selftest((cudaStream_t)stream, &e)) return CONVROT_ERR_UNSUPPORTED;
    return cuda_status(e);
}

}  // extern "C"
