// Diagnostics.
//
// A bounded wait that runs out.  One warp initialises an
// mbarrier that nothing will complete and waits on it with the same helper
// the inject kernel uses for its stages; the wait gives up after the given
// limit, the kernel records KVI_ERR_TIMEOUT and returns.  The tests use it to
// show that a wait which never completes ends with an error status the host
// reads, not a hang, and that the context stays usable.
//
// A streaming read by the SMs: every thread reads 16-byte words, grid-stride,
// with eight loads in flight, and the CTAs add what they read into one
// checksum (so that no load can be dropped).  Pointed at pinned host memory,
// its rate is the ceiling of the inject kernel's reads of a host-resident
// store, which use the same 16-byte loads (cp.async).
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

constexpr int kReadThreads = 512;
constexpr int kReadUnroll = 8;

__global__ void __launch_bounds__(kReadThreads) stream_read_kernel(const uint4 *src, uint64_t n16,
                                                                   unsigned long long *sum)
{
    const uint64_t stride = (uint64_t)gridDim.x * kReadThreads;
    uint64_t i = (uint64_t)blockIdx.x * kReadThreads + threadIdx.x;
    unsigned long long acc = 0;
    for (; i + (kReadUnroll - 1) * stride < n16; i += kReadUnroll * stride) {
        uint4 v[kReadUnroll];
#pragma unroll
        for (int u = 0; u < kReadUnroll; ++u) v[u] = __ldcg(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < kReadUnroll; ++u) acc += (unsigned long long)v[u].x + v[u].y + v[u].z + v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcg(src + i);
        acc += (unsigned long long)v.x + v.y + v.z + v.w;
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(sum, acc);
}

}  // namespace

cudaError_t launch_stream_read(const void *src, size_t bytes, int ctas_per_sm, uint64_t *sum, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(sum, 0, sizeof(uint64_t), s);
    if (e != cudaSuccess) return e;
    stream_read_kernel<<<(unsigned)(di.sms * ctas_per_sm), kReadThreads, 0, s>>>(
        static_cast<const uint4 *>(src), (uint64_t)(bytes / 16), reinterpret_cast<unsigned long long *>(sum));
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t *status, int64_t *elapsed_ns, cudaStream_t s)
{
    bounded_wait_kernel<<<1, 32, 0, s>>>(limit_ns, status, elapsed_ns);
    return cudaGetLastError();
}

}  // namespace kvi
