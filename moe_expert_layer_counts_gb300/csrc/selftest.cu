// selftest.cu -- self-test of the bounded mbarrier wait that every pipeline
// barrier of the library relies on.  A time-out here (or anywhere) is a
// status the host reads, never a trap or a fault: the waiting thread gives up
// at a global-timer deadline and the kernel returns normally.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// One CTA of 64 threads.  Thread 0 waits on a fresh barrier (one expected
// arrival); if `arrive`, thread 32 arrives after about 20 us.
__global__ void __launch_bounds__(64) bounded_wait_kernel(int arrive, uint64_t timeout_ns, int32_t* out) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint64_t t0 = ptx::globaltimer();
    if (threadIdx.x == 32 && arrive) {
        while (ptx::globaltimer() < t0 + 20000ull) __nanosleep(1000);  // ends: a fixed 20 us
        ptx::mbar_arrive(b);
    } else if (threadIdx.x == 0) {
        const bool ok = ptx::mbar_wait(b, 0, t0 + timeout_ns);
        out[0] = ok ? MOE_OK : MOE_ERR_TIMEOUT;
        out[1] = static_cast<int32_t>((ptx::globaltimer() - t0) / 1000ull);
    }
#else
    if (threadIdx.x == 0) out[0] = MOE_ERR_NO_KERNEL;
#endif
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int arrive, uint64_t timeout_ns, int32_t* out, cudaStream_t s) {
    bounded_wait_kernel<<<1, 64, 0, s>>>(arrive, timeout_ns, out);
    return cudaGetLastError();
}

}  // namespace moe
