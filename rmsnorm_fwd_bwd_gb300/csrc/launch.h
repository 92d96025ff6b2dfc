// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units (fwd.cu, bwd.cu). Internal: not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pool.h"

namespace rmsnorm {

// Arguments of every row kernel (forward and backward use disjoint subsets).
struct RowArgs {
    const void* x;
    const void* gamma;
    const void* dy;
    const float* rstd_in;  // backward: saved r per row
    void* y;               // forward output
    float* rstd_out;       // forward output
    void* dx;              // backward output
    float* ws;             // backward: dgamma partials [units][ldws] (LayerNorm: then dbeta partials)
    int64_t ldws;          // floats between partial rows: N rounded up to a multiple of 4, so that
                           // every partial row starts on a 16-byte boundary
    const void* beta;      // LayerNorm forward
    float* mean_out;       // LayerNorm forward output (may be null, as may rstd_out there)
    const float* mean_in;  // LayerNorm backward: saved mean per row
    const void* ddx;       // double backward: cotangent of dx [M rows, pitch ldddx]
    const void* ddg;       // double backward: cotangent of dgamma [N] (may be null: zero)
    void* d_dy;            // double backward output [M rows, pitch ldd_dy]; d_x goes to dx
    int64_t ldddx, ldd_dy;
    int64_t M;
    int N;
    int64_t ldx, ldy, lddy, lddx;  // row pitches in elements (>= N)
    float eps;
    int stages;            // TMA pipeline depth
    uint32_t* err;         // device error word
    RowPool pool;          // backward row pool (pool.head == 0: static assignment)
    unsigned long long* queue;  // the pool's queue word, after the partial rows:
                                // {call ticket (high 32 bits), segments taken}
    unsigned long long ticket;  // this call's ticket (low 32 bits used; consecutive
                                // calls in a process never share one)
    int pool_solo;              // forward pool, tuning: every CTA runs every segment
};

enum PathKind : int { kPathTma = 0, kPathScalar = 1, kPathRowVec = 2, kPathRagged = 3, kPathLanes = 4 };

// Most 16-byte vectors per thread on the row-vector path (256 threads).
constexpr int kRowVecMaxKv = 5;
// Row-vector grids are a multiple of this: rows r and r + 8 always start at the
// same 16-byte phase (a pitch is a whole number of 2-byte elements at least), so
// all rows of a persistent block (blockIdx.x + k * gridDim.x) share one phase.
constexpr int kRowVecPhases = 8;

// Thread caps (also the kernels' __launch_bounds__): a TMA-path slice is at most
// 1024 16-byte vectors, i.e. 256 threads x 4 vectors; the scalar path loops over
// the row with 256 threads.
constexpr int kTmaMaxThreads = 256;
// The double backward's single-CTA plans may take up to 16 warps (rows of up to
// 8192 elements at two vectors per thread, without a cluster barrier per row).
constexpr int kDbwdMaxThreads = 512;
// The RMSNorm backward's single-CTA plans for rows of 16-32 KB: 16 warps at up to
// four vectors per thread, instead of a two-CTA cluster.
constexpr int kWideRowThreads = 512;
constexpr int kWideRowMaxBytes = 32768;
// Narrow-row path (lanes.cu): blocks of 4 warps, a row per group of 4-32 lanes,
// aligned rows of at most kLaneMaxRowBytes.
constexpr int kLaneThreads = 128;
constexpr int kLaneMaxRowBytes = 2048;
// The ragged double backward may take up to 10 warps: fp32 rows of up to 16 KB
// then need at most four vectors per thread, 2-byte rows of up to 7672 elements
// three.
constexpr int kRaggedDbwdMaxThreads = 320;
constexpr int kScalarThreads = 256;
// Ring stages the pool kernel keeps row records for (bwd.cu, bwd_pool_kernel), and
// how many rows before the end of its head or segment a CTA takes its next segment
// (the take's round trip then overlaps those rows).
constexpr int kPoolMaxStages = 8;
constexpr int kPoolTakeAhead = 2;
// Queue words of the forward's row pool, one per call slot (fwd.cu).
constexpr unsigned kFwdQueueSlots = 4096;

// A launch shape chosen by the planner.
struct Plan {
    int path = kPathTma;
    int dtype = 0;
    int offset = 0;
    int cluster = 1;       // CTAs per cluster (TMA path)
    int threads = 0;       // threads per CTA
    int per_thread = 0;    // TMA: 16-byte vectors per thread; scalar: elements per thread
    int stages = 0;        // TMA pipeline depth
    size_t smem = 0;       // dynamic shared memory per CTA
    int64_t units = 0;     // clusters (TMA) or CTAs (scalar) = rows of dgamma partials
    int lanes = 0;         // narrow-row path: lanes per row (per_thread: vectors per lane)
    RowPool pool;          // RMSNorm backward, TMA path without clusters: the row pool
    int extra_threads = 0; // threads per CTA beyond `threads` (the pool kernel's producer warp)
};

// Rows of dgamma partials a plan writes, and the workspace bytes it needs: one
// partial row per CTA (cluster) and per pool segment, each ldws floats, then the
// pool's 16-byte queue word.
inline int64_t partial_rows(const Plan& p) { return p.units + p.pool.nseg; }

// Kernel entry for a plan (used for occupancy queries and attributes).
const void* fwd_kernel(const Plan& p);
const void* bwd_kernel(const Plan& p);
const void* rowvec_kernel(int pass, const Plan& p);  // pass 0 forward, 1 backward
const void* ragged_kernel(int pass, const Plan& p);  // TMA ring for rows off 16 bytes; pass 0 or 1
const void* ln_ragged_kernel(int pass, const Plan& p);  // the same for LayerNorm; pass 2 or 3
const void* ln_fwd_kernel(const Plan& p);             // LayerNorm (TMA or scalar path)
const void* ln_bwd_kernel(const Plan& p);
const void* ln_rowvec_kernel(int pass, const Plan& p);  // pass 2 forward, 3 backward
const void* lanes_kernel(int pass, const Plan& p);    // narrow rows, passes 0-4
const void* dbwd_kernel(const Plan& p);               // RMSNorm double backward (TMA, ragged or scalar path)
const void* dbwd_ragged_kernel_ptr(const Plan& p);    // its ragged TMA kernel
const void* dgamma_reduce_kernel_ptr(int dtype, int64_t units);  // launch shape depends on the row count

// Launch `k` with the plan's grid, block, shared memory and cluster shape, and
// programmatic stream serialization.
cudaError_t launch_rows(const void* k, const Plan& p, const RowArgs& a, cudaStream_t s);
// Column sums of the partial rows: dgamma from plane 0 of ws and, when dbeta is
// not null, dbeta from plane 1 (planes of units rows of ldws floats, one after the
// other; ldws a multiple of 4).
// Floats between the workspace's partial rows for rows of N elements.
inline int64_t workspace_pitch(int64_t N) { return (N + 3) / 4 * 4; }
inline size_t workspace_need(const Plan& p, int64_t N, int planes = 1) {
    return static_cast<size_t>(planes) * static_cast<size_t>(partial_rows(p)) *
               static_cast<size_t>(workspace_pitch(N)) * sizeof(float) +
           (p.pool.nseg > 0 ? 16 : 0);
}
// `queue`: the row pool's queue word to close once the row kernel is done (or null).
cudaError_t launch_dgamma_reduce(int dtype, const float* ws, int64_t units, int N, int64_t ldws, void* dgamma,
                                 cudaStream_t s, void* dbeta = nullptr, unsigned long long* queue = nullptr);

// Device address of the error word in the current context (nullptr on failure),
// looked up on every call.
uint32_t* device_error_word();
// Device address of the forward pool's queue word for a call slot (nullptr on
// failure), looked up on every call.
unsigned long long* fwd_queue_word(unsigned slot);

}  // namespace rmsnorm
