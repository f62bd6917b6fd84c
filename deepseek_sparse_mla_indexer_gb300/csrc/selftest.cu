// Self-test of the bounded wait every tensor-core kernel of the library uses:
// one block waits on an mbarrier that nothing arrives on, with a caller-given
// cycle budget, and must give up and report NSA_ERR_TIMEOUT instead of hanging.
#include "nsa_internal.cuh"
#include "sm100.cuh"

namespace nsa {
namespace {

__global__ void bounded_wait_kernel(int32_t *status, long long budget_cycles)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);  // one arrival expected; none will come
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0, budget_cycles)) set_status(status, NSA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace nsa

extern "C" nsa_status nsa_check_bounded_wait(int32_t *status_dev, long long budget_cycles, nsa_stream_t stream)
{
    if (!status_dev || budget_cycles < 1 || budget_cycles > 4000000000LL) return NSA_ERR_INVALID_ARG;
    nsa::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status_dev, budget_cycles);
    return nsa::launch_status();
}
