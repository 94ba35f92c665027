// Self-test of the bounded device waits used by every pipelined kernel: a
// kernel waits on an mbarrier phase that nothing completes, gives up after the
// given time and reports PCP_ERR_TIMEOUT through the status word, leaving the
// context usable. No fault, trap or endless loop is involved.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int32_t* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one arrival expected; none ever comes
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_warp(b, 0, &abort_flag, timeout_ns);
    if (!ok && threadIdx.x == 0) report_status(status, PCP_ERR_TIMEOUT);
}

}  // namespace
}  // namespace pcp

extern "C" int pcp_selftest_bounded_wait(int32_t* status, uint32_t timeout_us, pcp_stream_t stream) {
    if (!status || timeout_us < 1 || timeout_us > 1000000) return PCP_ERR_ARG;
    pcp::bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status,
                                                                                  (uint64_t)timeout_us * 1000ull);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        pcp::set_last_cuda_error(e);
        return PCP_ERR_CUDA;
    }
    return PCP_OK;
}
