// noalloc.cu -- rmsnorm_bwd_static_scratch: the backward pass for callers that
// cannot allocate device memory (see include/rmsnorm.h).
//
// The backward needs scratch for its per-block dgamma partial sums. Here that
// scratch is a fixed-size array in the library's own device memory instead of
// a caller buffer, and the call goes through the same validation, launch plan
// and kernels as rmsnorm_bwd.
#include <mutex>

#include "../../include/rmsnorm.h"
#include <cuda_runtime.h>

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchFloats = RMSNORM_STATIC_SCRATCH_BYTES / sizeof(float);

// One copy per device that loads the library, held until the process exits.
// In host code this name is only a stand-in: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device, looked up once per
// device (the first call on a device does the lookup).
rmsnorm_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return RMSNORM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return RMSNORM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return RMSNORM_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return RMSNORM_OK;
}

}  // namespace

extern "C" rmsnorm_status rmsnorm_bwd_static_scratch(const void* dy, const void* x, const void* gamma,
                                                     const float* rstd, void* dx, void* dgamma, int64_t M,
                                                     int64_t N, rmsnorm_dtype dtype, int offset,
                                                     rmsnorm_stream_t stream) {
    void* scratch = nullptr;
    const rmsnorm_status st = scratch_address(&scratch);
    if (st != RMSNORM_OK) return st;
    // rmsnorm_bwd rejects (RMSNORM_ERR_WORKSPACE) any shape whose partial sums
    // need more than RMSNORM_STATIC_SCRATCH_BYTES, before launching anything.
    // Every partial-sum row the column reduction reads is first written by the
    // row kernel of the same call, so nothing left over from an earlier call is
    // read and nothing needs clearing.
    return rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, offset, scratch,
                       RMSNORM_STATIC_SCRATCH_BYTES, stream);
}
