// Self-test of the pipeline's failure path: one CTA waits, with the same
// bounded mbarrier wait the tensor-core GEMM uses, on a barrier that nothing
// arrives on.  The wait must give up after its limit, record DEVERR_TIMEOUT in
// the device error word and let the kernel return, leaving the context usable.
// Checked builds add a kernel whose one bounds check fails (it touches no
// memory), for the reporting path of that build.
#include "common.cuh"
#include "convrot.h"
#include "internal.h"
#include "mbar.cuh"

namespace convrot {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Phase 0 never completes: no thread arrives on the barrier.
    (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
}

#ifdef CONVROT_CHECKED
__global__ void bounds_flag_kernel(int64_t extent) {
    // offset `extent` of a tensor holding `extent` elements: one past the end
    (void)CR_SPAN(extent, 1, extent);
}
#endif

}  // namespace

bool launch_bounds_flag_selftest(cudaStream_t st, cudaError_t *e) {
#ifdef CONVROT_CHECKED
    bounds_flag_kernel<<<1, 1, 0, st>>>(1);
    *e = cudaGetLastError();
    return true;
#else
    (void)st;
    *e = cudaSuccess;
    return false;
#endif
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, unsigned *err, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace convrot
