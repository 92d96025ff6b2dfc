/*
 * rmsnorm.h -- C ABI of librmsnorm.so: row-wise RMSNorm forward and backward on
 * one NVIDIA GB300 (sm_103a), hand-written CUDA kernels.
 *
 * Operation (page "Check an AI model calculation before accelerating it",
 * sections "Problem and reference formula" and "Why do we need a forward and a
 * backward pass?"; offset variant from the page "torchtitan kernel numerics
 * verification", section on the golden / reference / target implementations).
 * For each row i of an M x N matrix x:
 *
 *     r_i      = 1 / sqrt(mean_j(x_ij^2) + eps)
 *     y_ij     = x_ij * r_i * g_j            g = gamma, or (1 + gamma) with offset
 *     u_ij     = dy_ij * g_j
 *     dx_ij    = r_i * u_ij - x_ij * r_i^3 * mean_j(u_ij * x_ij)
 *     dgamma_j = sum_i dy_ij * x_ij * r_i    (a sum over rows, not a mean)
 *
 * Means divide by the logical N. All arithmetic is fp32 whatever the I/O dtype;
 * inputs are converted at load and each output element is rounded once, to
 * nearest-even, into the I/O dtype. dgamma is deterministic: fp32 partial sums,
 * each over a fixed set of rows added in row order, then one fixed-order column
 * reduction (no floating-point atomics), so repeated calls on the same device
 * with the same workspace size give identical bits. (The backward hands its last
 * rows out dynamically, in segments that each have their own partial sum, so
 * the sums do not depend on which thread block ran which rows.)
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers on the current CUDA device. The
 *     caller owns every buffer and the stream; the library allocates nothing
 *     and keeps no state between calls apart from launch-configuration caches
 *     and the device error word (rmsnorm_device_error).
 *   - Layout: dense row-major, row pitch = N elements. x, y, dy, dx, gamma and
 *     dgamma share the I/O dtype; rstd is float32[M]. Outputs must not overlap
 *     inputs.
 *   - Pointers must be aligned to their element size. Rows whose byte length is
 *     a multiple of 16 with 16-byte-aligned x/y/dy/dx/gamma take the TMA bulk-copy
 *     path (rows of at most 2 KB: a row per group of 4-32 lanes with 16-byte
 *     loads instead). When x and dy share their offset from a 16-byte boundary,
 *     other rows of up to 16 KB take a TMA path that copies each row's aligned
 *     span and masks its two end vectors, and rows of 16-20 KB a path with
 *     16-byte loads of that span; anything else takes a general path with
 *     scalar loads. All give results within the same correctness gate.
 *   - All calls are asynchronous on `stream` (NULL = legacy default stream).
 *     Validation happens on the host before any launch; when a call returns an
 *     error nothing was launched and no output was written. There is no
 *     fallback to another implementation, on the CPU or elsewhere.
 *   - 1 <= N <= RMSNORM_MAX_N; 0 <= M <= RMSNORM_MAX_M. M == 0 is valid: the
 *     forward does nothing and the backward writes dgamma = 0.
 *   - eps must be finite and > 0 (eps = 0 would turn an all-zero row into 0*inf).
 *   - offset must be 0 (y = x*r*gamma) or 1 (y = x*r*(1 + gamma)); dgamma has
 *     the same formula in both cases since d(1 + w)/dw = 1.
 */
#ifndef RMSNORM_H
#define RMSNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so that this header needs
 * no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* rmsnorm_stream_t;

#define RMSNORM_MAX_N 16384
#define RMSNORM_MAX_M 2147483647LL

typedef enum {
    RMSNORM_F32 = 0,  /* IEEE binary32 */
    RMSNORM_F16 = 1,  /* IEEE binary16 */
    RMSNORM_BF16 = 2  /* bfloat16 */
} rmsnorm_dtype;

typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_NULL = 1,        /* a required pointer is NULL */
    RMSNORM_ERR_SHAPE = 2,       /* M or N out of range */
    RMSNORM_ERR_DTYPE = 3,       /* dtype is not one of rmsnorm_dtype */
    RMSNORM_ERR_EPS = 4,         /* eps not finite or not > 0 */
    RMSNORM_ERR_ALIGN = 5,       /* a pointer is not aligned as required */
    RMSNORM_ERR_WORKSPACE = 6,   /* workspace smaller than rmsnorm_bwd_workspace_size */
    RMSNORM_ERR_UNSUPPORTED = 7, /* no kernel for this configuration */
    RMSNORM_ERR_CUDA = 8,        /* a CUDA runtime call or launch failed */
    RMSNORM_ERR_ARG = 9          /* another argument is invalid (offset not 0/1) */
} rmsnorm_status;

/*
 * Forward. Reads x[M*N] and gamma[N] (dtype), writes y[M*N] (dtype) and
 * rstd[M] (float32, r_i above; keep it for the backward).
 * x, gamma, y, rstd may be NULL only when M == 0.
 */
rmsnorm_status rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd,
                           int64_t M, int64_t N, float eps, rmsnorm_dtype dtype,
                           int offset, rmsnorm_stream_t stream);

/*
 * Bytes of device workspace rmsnorm_bwd needs for this shape on the CURRENT
 * device (it depends on the device's SM count). The workspace holds float32
 * dgamma partial sums, rows of N (padded to a multiple of 4 floats): one per
 * persistent block (or cluster) and, for the plans that hand their last rows out
 * from a queue, one per queued segment of rows plus the queue's 16 bytes (about
 * 1170 rows, 18 MiB, for bf16 65536 x 4096 on a 152-SM GB300). It must be 16-byte
 * aligned. Returns 0 when M == 0 or when an argument is invalid (rmsnorm_bwd then
 * reports the precise error). Host-only; launches nothing.
 */
size_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype);

/*
 * Backward. Reads dy[M*N], x[M*N], gamma[N] (dtype) and rstd[M] (float32 from
 * rmsnorm_fwd on the same x and eps; not validated), writes dx[M*N] and
 * dgamma[N] (dtype). Two launches on `stream`: the fused row kernel (dx and
 * per-block dgamma partials into `workspace`) and the column reduction.
 * `workspace` must hold at least rmsnorm_bwd_workspace_size(M, N, dtype)
 * bytes (it may be NULL when that is 0); a smaller one that still holds one
 * partial row per block is used without the row queue (every block then keeps a
 * fixed share of the rows: other partial sums, equally within the error bound,
 * and slower on large M). The workspace is scratch: its contents on entry are
 * ignored and on return are unspecified. Calls whose kernels overlap on the GPU
 * must not share a workspace.
 */
rmsnorm_status rmsnorm_bwd(const void* dy, const void* x, const void* gamma,
                           const float* rstd, void* dx, void* dgamma,
                           int64_t M, int64_t N, rmsnorm_dtype dtype, int offset,
                           void* workspace, size_t workspace_bytes,
                           rmsnorm_stream_t stream);

/*
 * Backward without any caller-provided or library-allocated device memory.
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot call cudaMalloc, for example a plugin whose host framework owns
 * all device memory and forbids allocation, or a process that has handed the
 * free device memory to a caching allocator and must not allocate outside it.
 *
 * Same arguments and results as rmsnorm_bwd, minus the workspace: the dgamma
 * partial sums go to a fixed array of RMSNORM_STATIC_SCRATCH_BYTES (16 MiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits. It is used as a workspace of that size (see rmsnorm_bwd:
 * without the row queue when the queue's partial rows do not fit); shapes whose
 * partial sums need more than that even then are rejected with
 * RMSNORM_ERR_WORKSPACE before anything is launched; on a 152-SM GB300 the
 * measured workloads need at most about 10 MiB without the queue.
 *
 * Every call looks up the array's device address in the current context (a
 * host-side runtime query, no allocation), so a device reset between calls is
 * harmless; the first call on a device also loads the library's code there,
 * so make that first call before any stream capture. No call allocates. All calls on a device share the one array: two
 * calls whose kernels overlap on the GPU (for example on different streams
 * without ordering between them) race on it and give wrong dgamma. The array
 * keeps the last call's partial sums and queue word; nothing in it has to start
 * at zero (a queue word from an earlier call carries that call's ticket and
 * starts a fresh queue).
 */
#define RMSNORM_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
rmsnorm_status rmsnorm_bwd_static_scratch(const void* dy, const void* x, const void* gamma,
                                          const float* rstd, void* dx, void* dgamma,
                                          int64_t M, int64_t N, rmsnorm_dtype dtype, int offset,
                                          rmsnorm_stream_t stream);

/*
 * Strided forms: the same operations on row-major tensors whose consecutive
 * rows are ld* elements apart (ld* >= N; the gaps between rows are neither read
 * nor written), e.g. a view of the first N columns of a wider matrix. With
 * ld* = N they are rmsnorm_fwd / rmsnorm_bwd. The fast paths need every row to
 * start on the same 16-byte boundary pattern: 16-byte aligned rows and pitches
 * take the TMA (or, up to 2 KB, the lane-group) path; x and dy rows at equal
 * offsets from a 16-byte boundary (equal pointer offsets, pitches equal modulo
 * 16 bytes) the ragged TMA or row-vector path; other combinations the general
 * path. The workspace of
 * rmsnorm_bwd_strided is sized by rmsnorm_bwd_workspace_size(M, N, dtype).
 * Extension of the pages' contract, which rejects non-contiguous inputs
 * ("Check an AI model calculation before accelerating it", section "Adapting
 * the kernel and moving to production", which names strides as the first
 * extension to build and test).
 */
rmsnorm_status rmsnorm_fwd_strided(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                                   float* rstd, int64_t M, int64_t N, float eps, rmsnorm_dtype dtype,
                                   int offset, rmsnorm_stream_t stream);
rmsnorm_status rmsnorm_bwd_strided(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                                   const void* gamma, const float* rstd, void* dx, int64_t lddx,
                                   void* dgamma, int64_t M, int64_t N, rmsnorm_dtype dtype, int offset,
                                   void* workspace, size_t workspace_bytes, rmsnorm_stream_t stream);

/* Static English text for a status code; never NULL. */
const char* rmsnorm_status_string(rmsnorm_status status);

/*
 * Device error word of the CURRENT device. Kernels that wait on an mbarrier
 * give up after a bounded number of polls, set bit 0 of this word and skip
 * their stores, so a hang becomes a reported error. Reading synchronizes the
 * device. *flags receives the word; clear != 0 resets it to 0.
 */
rmsnorm_status rmsnorm_device_error(uint32_t* flags, int clear);

/*
 * Self-test of the bounded waits behind rmsnorm_device_error: launches one
 * block on `stream` that waits, at most `polls` times (1 .. 2^21), on an
 * mbarrier that nothing ever completes. The wait gives up, the kernel sets
 * bit 0 of the device error word and returns; the CUDA context stays usable.
 * A diagnostic for the failure-detection path; no counterpart on the pages.
 */
rmsnorm_status rmsnorm_selftest_wait_timeout(uint32_t polls, rmsnorm_stream_t stream);

/*
 * Launch plan the library would use, as text (for logs and tests): the path
 * ("tma", "lanes", "ragged", "rowvec" or "scalar") and its shape, e.g.
 * "tma cluster=1 threads=256 vpt=2 stages=2 units=456 ...". pass: 0 = forward,
 * 1 = backward; 2 and 3: the LayerNorm forward and backward of layernorm.h; 4:
 * the double backward of rmsnorm_double_backward.h. aligned16: 1 if the data
 * pointers will be 16-byte aligned, 0 if not (x and dy -- and ddx -- sharing
 * their offset from a 16-byte boundary), 2 if they sit at different offsets.
 * Writes at most buf_len bytes including the terminating NUL. Host-only.
 */
rmsnorm_status rmsnorm_describe_plan(int pass, int64_t M, int64_t N, rmsnorm_dtype dtype,
                                     int aligned16, char* buf, size_t buf_len);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_H */
