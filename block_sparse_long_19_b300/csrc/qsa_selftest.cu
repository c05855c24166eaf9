// Self-test of the failure path every kernel of the library relies on: a
// bounded mbarrier wait that runs out reports QSA_ERR_TIMEOUT through the
// caller's status word and the kernel returns normally (no trap, no hang; the
// context stays usable).  The test waits on a phase that nothing completes.
#include "qsa_common.cuh"
#include "qsa_kernels.h"
#include "qsa.h"

namespace qsa {
namespace {

__global__ void selftest_wait_kernel(unsigned long long limit_ns, int arrive, int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) mbar_arrive(&bar);  // completes phase 0: the wait returns at once
        if (!mbar_wait(&bar, 0, limit_ns)) report(status, QSA_ERR_TIMEOUT);
    }
}

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_selftest_bounded_wait(int64_t limit_ns, int complete, int32_t *dev_status,
                                                void *stream) {
    if (!dev_status) return QSA_ERR_INVALID_ARG;
    if (limit_ns < 1 || limit_ns > 100000000) return QSA_ERR_INVALID_ARG;  // at most 0.1 s
    qsa::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(limit_ns), complete ? 1 : 0, dev_status);
    return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
