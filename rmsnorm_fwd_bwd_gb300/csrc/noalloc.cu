// noalloc.cu -- rmsnorm_bwd_static_scratch: the backward pass for callers that
// cannot allocate device memory (see include/rmsnorm.h).
//
// The backward needs scratch for its per-block dgamma partial sums. Here that
// scratch is a fixed-size array in the library's own device memory instead of
// a caller buffer, and the call goes through the same validation, launch plan
// and kernels as rmsnorm_bwd.
#include "../../include/rmsnorm.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchFloats = RMSNORM_STATIC_SCRATCH_BYTES / sizeof(float);

// One copy per device that loads the library, held until the process exits.
// In host code this name is only a stand-in: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

// Device address of g_bwd_scratch in the current context. Looked up on every
// call: the lookup is a host-side runtime query that allocates nothing, and an
// address kept from an earlier call would be stale after a device reset (the
// array then lives in a new context, possibly at another address). The first
// call on a device also loads the library's module there, which is why that
// first call should come before any stream capture.
rmsnorm_status scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return RMSNORM_ERR_CUDA;
    }
    *out = p;
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
    // rmsnorm_bwd runs without the row queue when the queue's partial rows do not
    // fit RMSNORM_STATIC_SCRATCH_BYTES, and rejects (RMSNORM_ERR_WORKSPACE) any
    // shape whose partial sums need more even then, before launching anything.
    // Every partial-sum row the column reduction reads is first written by the
    // row kernel of the same call, and a queue word left by an earlier call holds
    // that call's ticket, which starts a fresh queue: nothing needs clearing.
    return rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, offset, scratch,
                       RMSNORM_STATIC_SCRATCH_BYTES, stream);
}
