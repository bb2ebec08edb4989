// convrot_linear_fwd_noalloc: the forward of the ConvRot INT8 layer for
// callers that cannot hand the library a workspace.
//
// Some callers own no device allocator on the path where they run this layer:
// a host framework or plugin that only passes in pointers to memory it
// manages, a latency-critical loop where cudaMalloc (which synchronises the
// device) is not allowed, or a process with a fixed device-memory budget.  For
// them the activation codes and scales that convrot_linear_fwd keeps in the
// caller's workspace live here in one file-scope device array instead.
//
// The array is a fixed kScratchBytes per GPU that loads this library, held
// until the process exits.  All calls share it: two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// it and must be serialised by the caller.  Each call fully rewrites the part
// it reads (the quantizer writes every code and scale before the GEMM reads
// them), so nothing has to be cleared between calls.
#include <mutex>

#include "convrot.h"
#include "common.cuh"
#include "internal.h"

namespace {

// 64 MiB + 256 KiB: M * K * 2 bytes of codes plus M * 4 bytes of scales (each
// region rounded up to 256 bytes) must fit.  M = 8192 tokens at K = 4096 take
// 64 MiB of codes and 32 KiB of scales; the largest M at K = 4096 is 8219.
constexpr size_t kScratchBytes = (size_t(64) << 20) + (size_t(256) << 10);

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of the scratch array on the current device.  In host code
// the name g_fwd_scratch is only a host-side stand-in, so the address is
// looked up once per device with that device current and cached.  The cache
// is keyed by the device index alone: the library must not be used across a
// cudaDeviceReset (or any other replacement of the device's primary context),
// after which the cached address would no longer belong to the context.
int scratch_of_current_device(unsigned char **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CONVROT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // leave no error behind for the caller's next check
            return CONVROT_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_ptr[dev]);
    return CONVROT_OK;
}

}  // namespace

extern "C" {

size_t convrot_linear_fwd_noalloc_max_bytes(void) { return kScratchBytes; }

int convrot_linear_fwd_noalloc(const uint16_t *x, int64_t M, int64_t K, const int8_t *Wq, const float *scale_w,
                               int64_t N, int block, const uint16_t *bias, uint16_t *y, convrot_stream_t stream) {
    const bool block_ok = block == 8 || block == 16 || block == 32 || block == 64 || block == 128 || block == 256;
    if (!block_ok || K <= 0 || K % block != 0 || K % 16 != 0 || K > CONVROT_MAX_ROW || M < 0 || N < 0 ||
        N % 16 != 0 || M > INT32_MAX || N > INT32_MAX)
        return CONVROT_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return CONVROT_OK;
    if (!x || !Wq || !scale_w || !y || ((uintptr_t)x & 15u) || ((uintptr_t)Wq & 15u) || ((uintptr_t)y & 15u) ||
        ((uintptr_t)scale_w & 15u) || (bias && ((uintptr_t)bias & 15u)))
        return CONVROT_ERR_INVALID_ARG;
    const size_t codes = round256((size_t)M * (size_t)K * 2);
    if (codes + round256((size_t)M * 4) > kScratchBytes) return CONVROT_ERR_UNSUPPORTED;  // beyond the fixed scratch

    // Device checks and the error word come from the regular path.
    int rc = convrot_quantize_activation(x, 0, K, K, block, nullptr, nullptr, stream);
    if (rc != CONVROT_OK) return rc;
    unsigned char *scratch = nullptr;
    rc = scratch_of_current_device(&scratch);
    if (rc != CONVROT_OK) return rc;
    uint16_t *xq = reinterpret_cast<uint16_t *>(scratch);
    float *sx = reinterpret_cast<float *>(scratch + codes);
    rc = convrot_quantize_activation(x, M, K, K, block, xq, sx, stream);
    if (rc != CONVROT_OK) return rc;
    return convrot_gemm_dequant(xq, sx, M, K, Wq, scale_w, N, bias, y, stream);
}

}  // extern "C"
