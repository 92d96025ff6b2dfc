/*
 * rmsnorm_double_backward.h -- the gradient of the RMSNorm backward pass
 * (second-order autograd), in librmsnorm.so, one NVIDIA GB300 (sm_103a).
 *
 * Operation. The page "Check an AI model calculation before accelerating it"
 * (section "Adapting the kernel and moving to production") lists double
 * backward among the extensions its kernels do not validate. The backward of
 * rmsnorm.h maps (dy, x, g) to (dx, dgamma), g = gamma or (1 + gamma) with
 * offset. This entry point returns the gradients of
 *     L = sum_ij ddx_ij * dx_ij + sum_j ddgamma_j * dgamma_j
 * with respect to dy, x and gamma, r_i depending on x_i. For each row, with
 *     u = dy*g,  c = mean_j(u*x),  A = mean_j(ddx*x),  B = mean_j(ddx*u),
 *     D = mean_j(ddgamma*dy*x),  e = ddx - r^2*x*A:
 *     d_dy = g*r*e + r*x*ddgamma
 *     d_x  = r*ddgamma*dy - r^3*(c*ddx + u*A + x*(B + D)) + 3*r^5*c*A*x
 *     d_gamma_j = sum_i r_i*dy_ij*e_ij       (also the gradient of w with offset)
 * Arithmetic is fp32; each output element is rounded once into the I/O dtype;
 * d_gamma is deterministic (fixed-order reduction).
 *
 * Conventions are those of rmsnorm.h (device pointers, caller-owned buffers and
 * stream, asynchronous, host-side validation before any launch, no fallback,
 * same status and dtype codes, 1 <= N <= RMSNORM_MAX_N). Rows have explicit
 * pitches in elements (ld = N is dense). 16-byte aligned rows, pitches and
 * per-column pointers with N*sizeof(dtype) a multiple of 16 take the TMA path
 * (clusters for rows over 4096 elements); rows of ddx, dy and x at one 16-byte
 * phase (equal pointer phases, pitches equal modulo 16 bytes; outputs at any
 * phase) take the ragged TMA path up to 4100 fp32 or 7672 bf16 / fp16
 * elements; anything else the general path.
 */
#ifndef RMSNORM_DOUBLE_BACKWARD_H
#define RMSNORM_DOUBLE_BACKWARD_H

#include "rmsnorm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace rmsnorm_bwd_bwd needs (one plane of fp32 column
 * partials, one row per persistent block). 0 for M == 0 or invalid arguments. */
size_t rmsnorm_bwd_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype);

/*
 * ddx: [M rows, pitch ldddx], the cotangent of dx; ddgamma: [N], the cotangent
 * of dgamma, or NULL for zero; dy, x: the backward's inputs [M rows, pitches
 * lddy, ldx]; gamma: [N] (w with offset); rstd: float32[M] from rmsnorm_fwd on
 * the same x and eps. Outputs: d_dy [M rows, pitch ldd_dy], d_x [M rows, pitch
 * ldd_x], d_gamma [N], all in dtype. workspace: at least
 * rmsnorm_bwd_bwd_workspace_size(M, N, dtype) bytes, 16-byte aligned.
 * M == 0: writes d_gamma = 0 and reads nothing else.
 * Errors: RMSNORM_ERR_NULL, _SHAPE (M, N or a pitch), _DTYPE, _ARG (offset),
 * _ALIGN, _WORKSPACE, _UNSUPPORTED, _CUDA.
 */
rmsnorm_status rmsnorm_bwd_bwd(const void* ddx, int64_t ldddx, const void* ddgamma, const void* dy, int64_t lddy,
                               const void* x, int64_t ldx, const void* gamma, const float* rstd, void* d_dy,
                               int64_t ldd_dy, void* d_x, int64_t ldd_x, void* d_gamma, int64_t M, int64_t N,
                               rmsnorm_dtype dtype, int offset, void* workspace, size_t workspace_bytes,
                               rmsnorm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_DOUBLE_BACKWARD_H */
