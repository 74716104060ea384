// selftest.cu -- a self-test of the bounded waits every tensor-core kernel relies on.
//
// Each mbarrier wait in the library gives up after a time limit (tc_ptx.cuh), records
// GCL_DEV_WAIT_TIMEOUT in the device status word and returns, so that a lost copy or MMA
// completion ends as a status the host can read instead of a hung GPU.  This kernel exercises
// that path without any fault: one thread waits on an mbarrier that nothing arrives at.
#include "gcl_internal.cuh"
#include "tc_ptx.cuh"

namespace gcl {
namespace {

__global__ void wait_timeout_probe(int32_t *status) {
    __shared__ uint64_t bar;
    __shared__ int err;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        err = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &err, 1)) status_set(status, GCL_DEV_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace gcl

using namespace gcl;

extern "C" gcl_status_t gcl_selftest_wait_timeout(int32_t *dev_status, gcl_stream_t stream) {
    if (!dev_status) return fail(GCL_ERR_INVALID_ARG, "gcl_selftest_wait_timeout: dev_status is NULL");
    wait_timeout_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
    return cuda_check(cudaGetLastError(), "gcl_selftest_wait_timeout");
}
