// status.cu -- device status word helpers: reset (stream-ordered) and a self-test of the bounded
// wait that every kernel's mbarrier waits go through.
#include "common.cuh"
#include "kernels.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

__global__ void status_reset_kernel() {
    g_status = 0;
    g_abort = 0;
}

// One mbarrier that expects one arrival and never receives it: the bounded wait gives up after
// limit_ns and records CSA_ERR_TIMEOUT (and raises the abort flag) exactly as a stalled pipeline
// would in the attention or indexer kernels.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, limit_ns, nullptr)) set_timeout();
}

void launch_status_reset(cudaStream_t st) {
    status_reset_kernel<<<1, 1, 0, st>>>();
    count_launches(1);
}

void launch_wait_selftest(uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
    count_launches(1);
}

}  // namespace csa
