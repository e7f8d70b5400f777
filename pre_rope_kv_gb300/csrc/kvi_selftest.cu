// Diagnostic: a bounded wait that runs out.  One warp initialises an
// mbarrier that nothing will complete and waits on it with the same helper
// the inject kernel uses for its stages; the wait gives up after the given
// limit, the kernel records KVI_ERR_TIMEOUT and returns.  The tests use it to
// show that a wait which never completes ends with an error status the host
// reads, not a hang, and that the context stays usable.
#include <cuda_runtime.h>

#include "kvi_internal.cuh"
#include "kvi_sync.cuh"

namespace kvi {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(uint64_t limit_ns, int32_t *status, int64_t *elapsed_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) mbar_init(b, 1);  // one arrival expected; none will come
    __syncwarp();
    const uint64_t t0 = global_ns();
    const bool done = mbar_wait(b, 0, limit_ns);
    const uint64_t t1 = global_ns();
    if (threadIdx.x == 0) {
        if (!done) record_status(status, KVI_ERR_TIMEOUT);
        if (elapsed_ns) *elapsed_ns = (int64_t)(t1 - t0);
    }
}

}  // namespace

cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t *status, int64_t *elapsed_ns, cudaStream_t s)
{
    bounded_wait_kernel<<<1, 32, 0, s>>>(limit_ns, status, elapsed_ns);
    return cudaGetLastError();
}

}  // namespace kvi
