// sfa_selftest.cu -- a check of the failure path of the pipelined kernels:
// their every wait on an mbarrier is bounded, and a wait that gives up sets
// the CTA's abort flag (the other warps then leave their own waits early) and
// SFA_DEVSTAT_WAIT_TIMEOUT in the caller's status word, so the kernel returns
// and the context stays usable.  Here one CTA waits on a barrier that nothing
// arrives on, with the same wait routines the forward and backward kernels use:
// warp 0 as a producer lane does (mbar_wait), warp 1 as a consumer warp does
// (warp_wait, which must end through the abort flag).  No data is touched.
#include "sfa_internal.cuh"
#include "sfa_mma.cuh"
#include "sfa_ring.cuh"

namespace sfa {

namespace {

using namespace mma;
using namespace ring;

__global__ void __launch_bounds__(64) wait_selftest_kernel(unsigned* status) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0 && !mbar_wait(b, 0, &abort_flag)) {
            // the producer's failure path
            abort_flag = 1;
            if (status) atomicOr(status, SFA_DEVSTAT_WAIT_TIMEOUT);
        }
    } else {
        // a consumer warp: leaves through the abort flag (or its own limit)
        if (!warp_wait(b, 0, &abort_flag) && lane == 0 && status) atomicOr(status, SFA_DEVSTAT_WAIT_TIMEOUT);
    }
    __syncthreads();
    // nothing ever arrived: complete the phase so the barrier is left idle
    if (threadIdx.x == 0) mbar_arrive(b);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s) {
    wait_selftest_kernel<<<1, 64, 0, s>>>(status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace sfa
