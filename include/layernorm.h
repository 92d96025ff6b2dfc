/*
 * layernorm.h -- LayerNorm forward and backward in librmsnorm.so, on the same
 * kernel machinery as RMSNorm (rmsnorm.h), one NVIDIA GB300 (sm_103a).
 *
 * Operation. The page "torch.compile performance leap: optimizing LayerNorm
 * and RMSNorm kernels" (section 1.1) describes LayerNorm as normalising each
 * row by its mean and variance, then scaling by a learned weight gamma and
 * shifting by a learned bias beta; section 2 lists its three gradients (input,
 * weight, bias) and section 2.1 the fused backward that reduces along rows for
 * dx and along columns for dgamma and dbeta. The page prints no formula; this
 * library computes the standard one. For each row i of an M x N matrix x:
 *
 *     mu_i     = mean_j x_ij
 *     r_i      = 1 / sqrt(mean_j (x_ij - mu_i)^2 + eps)     (biased variance)
 *     xhat_ij  = (x_ij - mu_i) * r_i
 *     y_ij     = xhat_ij * gamma_j + beta_j
 *     u_ij     = dy_ij * gamma_j
 *     dx_ij    = r_i * (u_ij - mean_j u_ij - xhat_ij * mean_j(u_ij * xhat_ij))
 *     dgamma_j = sum_i dy_ij * xhat_ij
 *     dbeta_j  = sum_i dy_ij
 *
 * Arithmetic is fp32 whatever the I/O dtype; each output element is rounded
 * once, to nearest-even, into the I/O dtype. The variance is formed from
 * deviations about the mean (never as mean(x^2) - mean(x)^2). dgamma and dbeta
 * are deterministic (fixed-order reductions, no floating-point atomics).
 *
 * Conventions are those of rmsnorm.h: DEVICE pointers on the current device,
 * caller-owned buffers and stream, asynchronous on `stream`, host-side
 * validation before any launch (on error nothing was launched or written), no
 * fallback to another implementation, the same status codes and dtype codes,
 * 1 <= N <= RMSNORM_MAX_N, 0 <= M <= RMSNORM_MAX_M, eps finite and > 0.
 *
 * Layout: row-major with explicit row pitches in elements (ld >= N; ld = N is
 * dense). Rows whose pitches and pointers are 16-byte aligned and whose byte
 * length is a multiple of 16 take the TMA bulk-copy path (clusters of 2 or 4
 * CTAs for rows wider than 16 KB; rows of at most 2 KB a row per group of 4-32
 * lanes instead); rows whose x and dy share their offset from a 16-byte
 * boundary take a ragged TMA path (spans up to 16 KB) or a row-vector path
 * (16-20 KB); anything else takes a general path with scalar loads. Outputs
 * must not overlap inputs.
 */
#ifndef LAYERNORM_H
#define LAYERNORM_H

#include "rmsnorm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Forward. x: [M rows, pitch ldx] in dtype; gamma, beta: [N] in dtype;
 * y: [M rows, pitch ldy] in dtype (written); mean, rstd: float32[M] (written),
 * the row means mu_i and r_i saved for the backward. mean and rstd may each be
 * NULL when no backward will follow: they are then not written.
 * Errors: RMSNORM_ERR_NULL (x, gamma, beta or y NULL with M > 0),
 * RMSNORM_ERR_SHAPE (M, N or a pitch out of range), RMSNORM_ERR_DTYPE,
 * RMSNORM_ERR_EPS, RMSNORM_ERR_ALIGN (a pointer not aligned to its element
 * size), RMSNORM_ERR_UNSUPPORTED, RMSNORM_ERR_CUDA.
 */
rmsnorm_status layernorm_fwd(const void* x, int64_t ldx, const void* gamma, const void* beta, void* y,
                             int64_t ldy, float* mean, float* rstd, int64_t M, int64_t N, float eps,
                             rmsnorm_dtype dtype, rmsnorm_stream_t stream);

/*
 * Bytes of device workspace layernorm_bwd needs for M x N rows of `dtype`
 * (two planes of fp32 column partials, one row per persistent block: at most
 * a few MB at any M). 0 for M == 0 or invalid arguments. Host-only; queries
 * the current device.
 */
size_t layernorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype);

/*
 * Backward. dy: [M rows, pitch lddy]; x: [M rows, pitch ldx]; gamma: [N];
 * mean, rstd: float32[M] as written by layernorm_fwd on the same x, gamma,
 * beta and eps; dx: [M rows, pitch lddx] (written); dgamma, dbeta: [N] in
 * dtype (written). workspace: device scratch of at least
 * layernorm_bwd_workspace_size(M, N, dtype) bytes, 16-byte aligned, owned by
 * the caller and free for reuse once the call's work on `stream` is done.
 * M == 0: writes dgamma = dbeta = 0 and reads nothing else.
 * Errors: as layernorm_fwd, plus RMSNORM_ERR_WORKSPACE.
 */
rmsnorm_status layernorm_bwd(const void* dy, int64_t lddy, const void* x, int64_t ldx, const void* gamma,
                             const float* mean, const float* rstd, void* dx, int64_t lddx, void* dgamma,
                             void* dbeta, int64_t M, int64_t N, rmsnorm_dtype dtype, void* workspace,
                             size_t workspace_bytes, rmsnorm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LAYERNORM_H */
