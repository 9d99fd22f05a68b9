// Diagnostics of the library's failure path.  Every wait in the hot-path
// kernels is bounded: when its limit runs out the kernel records
// HS_ERR_TIMEOUT in the pool's sticky error word, abandons its work and
// returns, so the context stays usable.  hs_check_wait_timeout makes one such
// wait run out on purpose (an mbarrier that nothing completes), with the same
// bounded-wait routine, so that this path can be exercised without faulting
// or hanging anything.
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

}  // namespace

hs_status hs_check_wait_timeout(hs_pool *p, int64_t limit_cycles, cudaStream_t st) {
    if (!p || limit_cycles < 1000 || limit_cycles > hs::tc::kWaitCycles) return HS_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, st>>>((long long)limit_cycles, p->d.err);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
