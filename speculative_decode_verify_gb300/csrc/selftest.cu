// Self-test of the bounded waits every kernel of the library uses (failure detection without a fault):
// one thread waits on a shared-memory barrier that nothing completes, with the same wait routine as the
// attention kernels; it must give up after its time limit (or as soon as another warp raises the CTA's
// abort flag) and report VA_DEV_TIMEOUT in the status word, leaving the context usable.
#include <cuda_runtime.h>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

__global__ void bounded_wait_kernel(unsigned long long limit_ns, unsigned long long abort_after_ns,
                                    int32_t* dev_status, unsigned long long* elapsed_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);   // expects one arrival; none comes
        abort_flag = 0;
        ptx::mbar_init_fence();
    }
    __syncthreads();
    const uint64_t t0 = ptx::globaltimer_ns();
    if (threadIdx.x == 0) {
        const bool done = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, limit_ns);
        const uint64_t t = ptx::globaltimer_ns() - t0;
        if (!done && dev_status) atomicOr(dev_status, VA_DEV_TIMEOUT);
        if (elapsed_ns) *elapsed_ns = t;
    } else if (threadIdx.x == 32 && abort_after_ns > 0) {
        // raise the abort flag once abort_after_ns (<= limit_ns) have passed
        while (ptx::globaltimer_ns() - t0 < abort_after_ns) {
        }
        *reinterpret_cast<volatile int*>(&abort_flag) = 1;
    }
    __syncthreads();
}

}  // namespace va

extern "C" va_status va_selftest_bounded_wait(unsigned long long limit_ns, unsigned long long abort_after_ns,
                                              int32_t* dev_status, unsigned long long* elapsed_ns, va_stream stream) {
    if (limit_ns == 0 || limit_ns > VA_SELFTEST_MAX_WAIT_NS || abort_after_ns > limit_ns) return VA_INVALID_ARG;
    va::bounded_wait_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(limit_ns, abort_after_ns, dev_status, elapsed_ns);
    return cudaGetLastError() == cudaSuccess ? VA_OK : VA_CUDA_ERROR;
}
