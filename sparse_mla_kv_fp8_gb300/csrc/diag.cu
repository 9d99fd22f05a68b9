// Diagnostics of the library's failure path.  Every wait in the hot-path
// kernels is bounded: when its limit runs out the kernel records
// HS_ERR_TIMEOUT in the pool's sticky error word, abandons its work and
// returns, so the context stays usable.  hs_check_wait_timeout makes one such
// wait run out on purpose (an mbarrier that nothing completes), with the same
// bounded-wait routine, so that this path can be exercised without faulting
// or hanging anything.
//
// hs_host_read_probe measures the host link the miss copy uses: a grid of
// threads reads pinned host memory through its device mapping (zero-copy, the
// same 16-byte loads as the miss copy, four in flight per thread) and writes
// it to device memory.
#include "hs_internal.h"
#include "tc.cuh"

namespace {

__global__ void wait_timeout_kernel(long long limit, int32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        hs::tc::mbar_init(&bar, 1);  // one arrival expected; none ever comes
        hs::tc::fence_barrier_init();
    }
    __syncthreads();
    hs::tc::mbar_wait_limit(&bar, 0, err, limit);
}

__global__ void __launch_bounds__(256) host_read_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, size_t n16) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; k++) v[k] = src[i + k * stride];
#pragma unroll
        for (int k = 0; k < 4; k++) dst[i + k * stride] = v[k];
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace

hs_status hs_host_read_probe(const void *host_src, void *dev_dst, size_t bytes, int32_t ctas,
                             cudaStream_t st) {
    if (!host_src || !dev_dst || bytes == 0 || bytes % 16 || ((uintptr_t)host_src & 15) ||
        ((uintptr_t)dev_dst & 15) || ctas < 0 || ctas > 64 * hs::kNumSMs)
        return HS_ERR_INVALID_ARG;
    void *src = nullptr;
    if (cudaHostGetDevicePointer(&src, const_cast<void *>(host_src), 0) != cudaSuccess || !src) {
        cudaGetLastError();
        return HS_ERR_INVALID_ARG;  // not pinned host memory
    }
    const int grid = ctas ? ctas : 4 * hs::kNumSMs;
    host_read_kernel<<<grid, 256, 0, st>>>((const uint4 *)src, (uint4 *)dev_dst, bytes / 16);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status hs_check_wait_timeout(hs_pool *p, int64_t limit_cycles, cudaStream_t st) {
    if (!p || limit_cycles < 1000 || limit_cycles > hs::tc::kWaitCycles) return HS_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, st>>>((long long)limit_cycles, p->d.err);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
