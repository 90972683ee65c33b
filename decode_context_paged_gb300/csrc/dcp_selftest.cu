// dcp_selftest.cu -- dcp_selftest_wait_timeout: the device-side failure path, exercised on purpose.
//
// Every pipeline wait in the library (TMA completions, MMA commits, the softmax hand-offs) goes
// through mbar_wait, which gives up after a wall-time limit, raises the CTA's abort flag and
// ORs DCP_DEVERR_TIMEOUT into the caller's device error word instead of spinning forever.  This
// entry point runs that wait on an mbarrier nothing ever completes, so that a test can watch
// the limit expire, read the status on the host and go on using the context.  Nothing faults,
// traps or hangs: the one waiting thread returns after limit_ns.
#include <cuda_runtime.h>

#include "dcp_internal.h"
#include "dcp_ptx.cuh"

namespace dcp {
namespace {

__global__ void wait_selftest_kernel(uint64_t limit_ns, int32_t *dev_error, int32_t *out_ok) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 of a barrier that expects one arrival, which never comes
        const bool ok = mbar_wait(&bar, 0, &abort_flag, dev_error, limit_ns);
        *out_ok = ok ? 1 : 0;
    }
}

}  // namespace
}  // namespace dcp

extern "C" int dcp_selftest_wait_timeout(uint64_t limit_ns, int32_t *dev_error, int32_t *out_ok,
                                         dcp_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull || !dev_error || !out_ok) return DCP_ERR_INVALID_ARG;
    dcp::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, dev_error, out_ok);
    return cudaGetLastError() == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}
