// Self-test of the bounded-wait path shared by every kernel of the library:
// one CTA waits on an mbarrier that nobody arrives on. The wait gives up after
// its time bound, records its site in the workspace error word and the kernel
// returns, leaving the context usable.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int32_t kSelftestSite = 0x7F;

__global__ void selftest_timeout_kernel(int32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none will come
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, kSelftestSite);
}

}  // namespace

cudaError_t launch_selftest_timeout(int32_t* err, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace da
