// selftest.cu -- exercises the bounded mbarrier wait that every pipelined
// kernel uses, on a barrier that nothing ever completes.
#include "../../include/rmsnorm.h"
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

// One thread initialises an mbarrier expecting one arrival that never comes,
// then waits for it with the given poll limit. The wait must give up, set the
// timeout bit in the device error word and let the kernel finish.
__global__ void wait_timeout_kernel(uint32_t polls, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        mbar_wait_bounded(smem_u32(&bar), 0, err, polls);
    }
}

}  // namespace rmsnorm

extern "C" rmsnorm_status rmsnorm_selftest_wait_timeout(uint32_t polls, rmsnorm_stream_t stream) {
    if (polls == 0 || polls > (1u << 21)) return RMSNORM_ERR_ARG;
    uint32_t* err = rmsnorm::device_error_word();
    if (!err) return RMSNORM_ERR_CUDA;
    rmsnorm::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(polls, err);
    return cudaGetLastError() == cudaSuccess ? RMSNORM_OK : RMSNORM_ERR_CUDA;
}
