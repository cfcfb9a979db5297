// Self-test of the bounded device waits (failure detection without a GPU
// fault). The tensor-core kernels wait on mbarriers for TMA copies and MMAs.
// Each such wait gives up after a time limit, sets SSA_DEV_WAIT_LIMIT in
// *dev_status, stops the block's other roles and returns, so a copy or MMA
// that never completes costs an error status, not a hung GPU. This kernel
// takes the same path on purpose. One thread waits on an mbarrier that
// nothing arrives on, with the production wait helper, until the limit runs
// out.
#include "sm100.cuh"
#include "trace.h"

namespace ssa {

__global__ void wait_limit_selftest_kernel(int32_t* dev_status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);   // one arrival would complete phase 0; none comes
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) sm100::mbar_wait_bounded(&bar, 0, &abort_flag, dev_status, limit_ns);
}

}  // namespace ssa

extern "C" ssa_status ssa_selftest_wait_limit(int32_t* dev_status, uint64_t limit_ns,
                                              void* stream) {
    if (!dev_status || (reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0)
        return SSA_ERR_INVALID;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return SSA_ERR_INVALID;   // at most one second
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ssa::TraceLaunch tr("wait_limit_selftest", s);
    ssa::wait_limit_selftest_kernel<<<1, 32, 0, s>>>(dev_status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}
