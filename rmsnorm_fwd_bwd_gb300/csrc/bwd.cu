// bwd.cu -- RMSNorm backward kernels.
//
// Per row, with r the saved forward value and g = gamma (or 1 + w):
//     u = dy * g;   c = sum_j(u_j * x_j) / N;   dx = r * u - x * r^3 * c
// and, per column, dgamma_j = sum over rows of (dy_j * x_j) * r
// (page "Check an AI model calculation before accelerating it", sections
// "Input backward pass: keep the right N", "Where does the cube of r come
// from?" and "Reducing dgamma without a write race").
//
// The row pass is one fused kernel: x and dy are read once (TMA ring as in the
// forward), dx is written, and each persistent block keeps fp32 dgamma
// accumulators for its fixed columns in registers across its rows. In
// bwd_tma_kernel every block (cluster) takes a fixed share of the rows and writes
// one row of partials at the end; bwd_pool_kernel (the row pool of pool.h) takes a
// fixed head of rows, then segments of rows from a queue, and writes one partial
// row per head and per segment. A second kernel sums the partial rows per column
// in a fixed order, so dgamma is deterministic and no floating-point atomics are
// used (the page's own reason for private partial rows followed by a column
// pass). The workspace is a few rows per SM of N floats instead of one row of
// partials per input row.
#include "device.cuh"
#include "launch.h"
#include "pool.cuh"

namespace rmsnorm {

// Minimum resident blocks passed to __launch_bounds__ (0: none). Left alone,
// ptxas compiles the fp32 4-vector instance into 64 registers with spills; a
// floor of 2 blocks (at most 128 registers) gives it 96 and no spills.
template <int DT, int VPT> struct BwdMinBlocks { static constexpr int value = 0; };
template <> struct BwdMinBlocks<kF32, 4> { static constexpr int value = 2; };
// Block-size bound: the unsplit instances of up to four vectors per thread may
// take kWideRowThreads threads (one block per row of up to 32 KB instead of a
// two-CTA cluster); their register cap is then 128, as the floor above gives the
// fp32 4-vector instance.
template <int DT, int VPT, bool CLUSTER> struct BwdTmaBounds {
    static constexpr bool wide = !CLUSTER && VPT <= 4;
    static constexpr int threads = wide ? kWideRowThreads : kTmaMaxThreads;
    static constexpr int min_blocks = wide ? (BwdMinBlocks<DT, VPT>::value ? 1 : 0) : BwdMinBlocks<DT, VPT>::value;
};

template <int DT, int VPT, bool OFFSET, bool CLUSTER>
__global__ void __launch_bounds__(BwdTmaBounds<DT, VPT, CLUSTER>::threads, (BwdTmaBounds<DT, VPT, CLUSTER>::min_blocks))
    bwd_tma_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const uint32_t crank = CLUSTER ? cluster_rank() : 0u;
    const uint32_t csize = CLUSTER ? cluster_size() : 1u;
    const int64_t cid = CLUSTER ? static_cast<int64_t>(cluster_id()) : static_cast<int64_t>(blockIdx.x);
    const int64_t ncl = CLUSTER ? static_cast<int64_t>(cluster_count()) : static_cast<int64_t>(gridDim.x);

    const int ns = a.N / static_cast<int>(csize);
    const int nvec = ns / VEC;
    const uint32_t slice_bytes = static_cast<uint32_t>(ns) * E::kBytes;
    const uint32_t stage_bytes = 2 * slice_bytes;  // x slice, then dy slice
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
    const size_t dx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const int S = a.stages;

    // shared memory: ring | gamma slice in fp32 | mbarriers | warp partials [2][32] | abort flag
    unsigned char* ring = smem;
    float* gsm = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(gsm + ns);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;
    const size_t slice_off = static_cast<size_t>(crank) * slice_bytes;
    const char* xsl = static_cast<const char*>(a.x) + slice_off;
    const char* dysl = static_cast<const char*>(a.dy) + slice_off;
    char* dxsl = static_cast<char*>(a.dx) + slice_off;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_wait();  // inputs may come from the previous kernel on the stream
    // the first rows' copies go out before the per-column set-up below, so the
    // ring fills while gamma is being loaded
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t j, const unsigned char* st, uint32_t bar) {
        const size_t r = static_cast<size_t>(cid + j * ncl);
        mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_g2s_in(smem_u32(st), xsl + r * x_pitch, slice_bytes, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
        bulk_g2s_in(smem_u32(st + slice_bytes), dysl + r * dy_pitch, slice_bytes, bar, pol,
                    a.dy, a.M, a.lddy, a.N, E::kBytes, a.err);
    };
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) issue(j, ring + j * stage_bytes, smem_u32(&full[j]));
    }

    // gamma slice widened once (offset variant: 1 + w) into shared memory, as
    // VEC/4 planes of float4 so that a warp reads 512 consecutive bytes per plane
    float4* gsm4 = reinterpret_cast<float4*>(gsm);
    {
        const uint4* gs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.gamma) + slice_off);
        for (int idx = tid; idx < nvec; idx += nt) {
            float w[VEC];
            E::unpack(__ldg(gs + idx), w);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                float4 f = OFFSET ? make_float4(1.0f + w[q], 1.0f + w[q + 1], 1.0f + w[q + 2], 1.0f + w[q + 3])
                                  : make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
                gsm4[(q / 4) * nvec + idx] = f;
            }
        }
    }
    float acc[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;

    __syncthreads();
    if (CLUSTER) cluster_sync();

    // saved r, 32 rows per warp-wide load, fetched 32 rows ahead of use
    auto rstd_at = [&](int64_t jj) -> float {
        return jj < nrows ? __ldg(a.rstd_in + cid + jj * ncl) : 0.f;
    };
    float r_cur = rstd_at(lane);
    float r_next = rstd_at(32 + lane);

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = cid + j * ncl;
        const unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
        if ((j & 31) == 0 && j > 0) {
            r_cur = r_next;
            r_next = rstd_at(j + 32 + lane);
        }
        const float r = __shfl_sync(0xffffffffu, r_cur, static_cast<int>(j & 31));

        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        float xf[VPT][VEC], uf[VPT][VEC];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            float df[VEC], g[VEC];
            if (idx < nvec) {
                E::unpack(*reinterpret_cast<const uint4*>(st + idx * 16), xf[v]);
                E::unpack(*reinterpret_cast<const uint4*>(st + slice_bytes + idx * 16), df);
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    const float4 f = gsm4[(q / 4) * nvec + idx];
                    g[q] = f.x; g[q + 1] = f.y; g[q + 2] = f.z; g[q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) xf[v][e] = df[e] = g[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                uf[v][e] = __fmul_rn(df[e], g[e]);
                if (e & 1) p1 = fmaf(uf[v][e], xf[v][e], p1); else p0 = fmaf(uf[v][e], xf[v][e], p0);
                acc[v][e] = fmaf(__fmul_rn(df[e], xf[v][e]), r, acc[v][e]);
            }
        }
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(p0 + p1);
        if (lane == 0) redb[warp] = wsum;
        if (CLUSTER) cluster_sync(); else __syncthreads();
        if (!aborted && *abort_flag) {
            aborted = true;
            abort_row = j;
        }

        if (tid == 0 && !aborted && j + S < nrows) {
            fence_proxy_async_smem();
            issue(j + S, st, smem_u32(&full[s]));
        }
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }

        float t = 0.f;
        if (!CLUSTER) {
            if (lane < nwarps) t = redb[lane];
        } else if (lane < nwarps * static_cast<int>(csize)) {
            t = dsmem_ld_f32(dsmem_map(smem_u32(redb + lane % nwarps), lane / nwarps));
        }
        t = warp_allsum(t);
        const float c = t / static_cast<float>(a.N);
        // dx = r*u - x*k with k = r^3 * c, as one fused multiply-add per element
        const float k = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), c);

        if (!aborted) {
            char* dxrow = dxsl + static_cast<size_t>(row) * dx_pitch;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nt + tid;
                if (idx < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf(-xf[v][e], k, __fmul_rn(r, uf[v][e]));
                    stg128(dxrow + idx * 16, E::pack(o));
                }
            }
        }
    }

    griddep_launch_dependents();
    // one row of dgamma partials per cluster: ws[cid][crank*ns + ...]
    if (!aborted) {
        float* wrow = a.ws + static_cast<size_t>(cid) * a.ldws + static_cast<size_t>(crank) * ns;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            if (idx < nvec) {
#pragma unroll
                for (int q = 0; q < VEC; q += 4)
                    *reinterpret_cast<float4*>(wrow + idx * VEC + q) =
                        make_float4(acc[v][q], acc[v][q + 1], acc[v][q + 2], acc[v][q + 3]);
            }
        }
    }
    if (CLUSTER) cluster_sync();
    if (aborted && tid == 0) {
        const int64_t end = abort_row + S < nrows ? abort_row + S : nrows;
        for (int64_t j = abort_row; j < end; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), static_cast<uint32_t>((j / S) & 1), a.err, 1u << 16);
    }
}

// Backward row kernel with the row pool of pool.h (no clusters), formulas as in
// bwd_tma_kernel. CTA b first takes rows b + j * G, j < a.pool.head (dgamma
// partial row b), then segments of consecutive rows from the queue (partial row
// G + k for segment k); CTA 0 opens the queue for this call as it starts.
//
// The CTA is a.threads consumer threads plus one producer warp. The producer's
// lane 0 runs the ring ahead of the consumers: for each stage it waits until every
// consumer warp has released the stage's previous row (the `empty` barrier, one
// arrival per consumer warp), decides the next row (head, then queue; the take is
// issued kPoolTakeAhead rows before it is needed), records the row and the partial
// row to write after it in shared memory, and issues the TMA copies of x and dy
// and a 4-byte cp.async of the row's r, all completing on the stage's `full`
// barrier (two arrivals: the copies' expect_tx and the cp.async). A stage with no
// row (queue empty) is completed by plain arrivals and ends both loops. The
// consumers' only barrier per row is a named barrier among themselves (the row
// sum), so the producer's bookkeeping never delays a row.
// At most 128 registers (no spills at up to four vectors per thread): three CTAs of
// 128 consumer threads and the producer warp then fit an SM.
template <int DT, int VPT, bool OFFSET>
__global__ void __maxnreg__(128) bwd_pool_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int64_t stage_row[kPoolMaxStages];
    __shared__ int64_t stage_unit[kPoolMaxStages];
    __shared__ float stage_r[kPoolMaxStages];
    __shared__ uint64_t empty[kPoolMaxStages];

    const int tid = threadIdx.x;
    const int nc = blockDim.x - 32;  // consumer threads
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int ncw = nc >> 5;         // consumer warps; the producer is warp ncw
    const int64_t G = gridDim.x;

    const int nvec = a.N / VEC;
    const uint32_t row_bytes = static_cast<uint32_t>(a.N) * E::kBytes;
    const uint32_t stage_bytes = 2 * row_bytes;  // x row, then dy row
    const int S = a.stages;

    // shared memory: ring | gamma in fp32 | full barriers | warp partials [2][32] | abort flag
    unsigned char* ring = smem;
    float* gsm = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(gsm + a.N);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 2);
            mbar_init(smem_u32(&empty[s]), static_cast<uint32_t>(ncw));
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();  // inputs may come from the previous kernel on the stream

    if (warp == ncw) {
        // ---------------- producer ----------------
        if (lane != 0) return;
        const uint32_t ticket = static_cast<uint32_t>(a.ticket);
        const uint64_t pol = l2_evict_first_policy();
        const char* xb = static_cast<const char*>(a.x);
        const char* dyb = static_cast<const char*>(a.dy);
        const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
        const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
        PoolRows rows;
        int64_t issued = 0;
        bool aborted = false;
        for (;; ++issued) {
            const int s = static_cast<int>(issued % S);
            const int64_t round = issued / S;
            if (round > 0 &&
                !mbar_wait_or_abort(smem_u32(&empty[s]), static_cast<uint32_t>((round - 1) & 1), a.err,
                                    abort_flag)) {
                aborted = true;
                break;
            }
            int64_t unit;
            const int64_t row = rows.next(a, G, ticket, unit);
            stage_row[s] = row;
            stage_unit[s] = unit;
            const uint32_t bar = smem_u32(&full[s]);
            if (row < 0) {
                mbar_arrive_n(bar, 2);
                break;
            }
            unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
            cp_async4(smem_u32(&stage_r[s]), a.rstd_in + row);
            cp_async_arrive_noinc(bar);
            mbar_arrive_expect_tx(bar, stage_bytes);
            bulk_g2s_in(smem_u32(st), xb + static_cast<size_t>(row) * x_pitch, row_bytes, bar, pol, a.x, a.M,
                        a.ldx, a.N, E::kBytes, a.err);
            bulk_g2s_in(smem_u32(st + row_bytes), dyb + static_cast<size_t>(row) * dy_pitch, row_bytes, bar, pol,
                        a.dy, a.M, a.lddy, a.N, E::kBytes, a.err);
            if (issued == 0 && blockIdx.x == 0) pool_open(a.queue, ticket, a.pool.nseg, G, a.err);
        }
        if (aborted) {
            // the consumers gave up: wait for the copies of the stages issued last
            // (at most S of them may still be in flight) before the CTA exits
            for (int64_t i = issued - S < 0 ? 0 : issued - S; i < issued; ++i)
                if (stage_row[i % S] >= 0)
                    mbar_wait_bounded(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), a.err,
                                      1u << 16);
        }
        return;
    }

    // ---------------- consumers ----------------
    // gamma widened once (offset variant: 1 + w), VEC/4 planes of float4
    float4* gsm4 = reinterpret_cast<float4*>(gsm);
    {
        const uint4* gs = reinterpret_cast<const uint4*>(a.gamma);
        for (int idx = tid; idx < nvec; idx += nc) {
            float w[VEC];
            E::unpack(__ldg(gs + idx), w);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                float4 f = OFFSET ? make_float4(1.0f + w[q], 1.0f + w[q + 1], 1.0f + w[q + 2], 1.0f + w[q + 3])
                                  : make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
                gsm4[(q / 4) * nvec + idx] = f;
            }
        }
    }
    float acc[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;
    named_barrier_sync(1, nc);  // gamma planes are visible to every consumer

    char* dxb = static_cast<char*>(a.dx);
    const size_t dx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    // partial rows are read back by the column reduce right after this kernel:
    // keep them in L2 while the ring streams x and dy through it (bf16 65536x4096
    // backward 246.6 -> 242.8 us, fp16 16384x8192 133.4 -> 133.2)
    const uint64_t keep = l2_evict_last_policy();
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0;; ++j) {
        if (!mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;
        const int64_t row = stage_row[s];
        const int64_t unit = stage_unit[s];
        if (row < 0) break;  // the queue is empty (every consumer reads the same stage)
        const unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
        const float r = stage_r[s];

        float xf[VPT][VEC], uf[VPT][VEC];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nc + tid;
            float df[VEC], g[VEC];
            if (idx < nvec) {
                E::unpack(*reinterpret_cast<const uint4*>(st + idx * 16), xf[v]);
                E::unpack(*reinterpret_cast<const uint4*>(st + row_bytes + idx * 16), df);
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    const float4 f = gsm4[(q / 4) * nvec + idx];
                    g[q] = f.x; g[q + 1] = f.y; g[q + 2] = f.z; g[q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) xf[v][e] = df[e] = g[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                uf[v][e] = __fmul_rn(df[e], g[e]);
                if (e & 1) p1 = fmaf(uf[v][e], xf[v][e], p1); else p0 = fmaf(uf[v][e], xf[v][e], p0);
                acc[v][e] = fmaf(__fmul_rn(df[e], xf[v][e]), r, acc[v][e]);
            }
        }
        // this warp is done with the stage: the producer may refill it once every
        // consumer warp has said so
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(p0 + p1);
        if (lane == 0) redb[warp] = wsum;
        named_barrier_sync(1, nc);
        if (*abort_flag) break;  // every consumer reads the flag after the same barrier

        float t = lane < ncw ? redb[lane] : 0.f;
        t = warp_allsum(t);
        const float c = t / static_cast<float>(a.N);
        // dx = r*u - x*k with k = r^3 * c, as one fused multiply-add per element
        const float k = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), c);
        char* dxrow = dxb + static_cast<size_t>(row) * dx_pitch;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nc + tid;
            if (idx < nvec) {
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = fmaf(-xf[v][e], k, __fmul_rn(r, uf[v][e]));
                stg128(dxrow + idx * 16, E::pack(o));
            }
        }
        // the last row of a head or a segment: its partial row, then fresh sums
        if (unit >= 0) {
            float* wrow = a.ws + static_cast<size_t>(unit) * a.ldws;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nc + tid;
                if (idx < nvec) {
#pragma unroll
                    for (int q = 0; q < VEC; q += 4)
                        stg_f4_hint(wrow + idx * VEC + q, acc[v][q], acc[v][q + 1], acc[v][q + 2], acc[v][q + 3], keep);
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;
            }
        }
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
    griddep_launch_dependents();
}

// General path: any N, any element alignment. One CTA per row (persistent);
// thread t owns columns t, t + nt, ...; two passes over the row (the second is
// served by L1/L2); dgamma accumulators live in shared memory indexed by column
// (each column is touched by one thread only).
template <int DT, bool OFFSET>
__global__ void __launch_bounds__(kScalarThreads) bwd_scalar_kernel(const RowArgs a) {
    using E = Elem<DT>;
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);  // [N]
    __shared__ float red[2][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    griddep_wait();

    for (int c = tid; c < N; c += nt) acc[c] = 0.f;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t base = row * a.ldx;
        const int64_t dbase = row * a.lddy;
        const int64_t obase = row * a.lddx;
        const float r = __ldg(a.rstd_in + row);
        // pass 1: sum of u*x, and this row's dgamma terms
        float p0 = 0.f, p1 = 0.f;
        int col = tid;
        for (; col + nt < N; col += 2 * nt) {
            const float x0 = E::ld(a.x, base + col), x1 = E::ld(a.x, base + col + nt);
            const float d0 = E::ld(a.dy, dbase + col), d1 = E::ld(a.dy, dbase + col + nt);
            const float w0 = E::ld(a.gamma, col), w1 = E::ld(a.gamma, col + nt);
            p0 = fmaf(__fmul_rn(d0, OFFSET ? 1.0f + w0 : w0), x0, p0);
            p1 = fmaf(__fmul_rn(d1, OFFSET ? 1.0f + w1 : w1), x1, p1);
            acc[col] = fmaf(__fmul_rn(d0, x0), r, acc[col]);
            acc[col + nt] = fmaf(__fmul_rn(d1, x1), r, acc[col + nt]);
        }
        for (; col < N; col += nt) {
            const float x0 = E::ld(a.x, base + col);
            const float d0 = E::ld(a.dy, dbase + col);
            const float w0 = E::ld(a.gamma, col);
            p0 = fmaf(__fmul_rn(d0, OFFSET ? 1.0f + w0 : w0), x0, p0);
            acc[col] = fmaf(__fmul_rn(d0, x0), r, acc[col]);
        }
        const float ws = warp_allsum(p0 + p1);
        if (lane == 0) red[parity][warp] = ws;
        __syncthreads();
        float t = lane < nwarps ? red[parity][lane] : 0.f;
        t = warp_allsum(t);
        const float c = t / static_cast<float>(N);
        const float k = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), c);  // dx = r*u - x*k
        // pass 2: the row again (now in L1/L2), dx
#pragma unroll 4
        for (int cc = tid; cc < N; cc += nt) {
            const float xv = E::ld(a.x, base + cc);
            const float dv = E::ld(a.dy, dbase + cc);
            const float w = E::ld(a.gamma, cc);
            const float u = __fmul_rn(dv, OFFSET ? 1.0f + w : w);
            E::st(a.dx, obase + cc, fmaf(-xv, k, __fmul_rn(r, u)));
        }
    }
    griddep_launch_dependents();
    if (blockIdx.x < a.M) {
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
        for (int c = tid; c < N; c += nt) wrow[c] = acc[c];
    }
}

// dgamma[j] = sum_{p < units} ws[p][j] in a fixed order, without atomics.
// A block owns an 8-column tile (two float4 lanes) of the partial rows and
// 16 * WARPS row lanes: lane (cq, rq) of warp w owns columns 4cq..4cq+3 and rows
// ry = 16w + rq, ry + 16 * WARPS, ... (8 warps; 16 when there are more than 1024
// partial rows, so that one batch of loads still covers them). Partial rows are ldws floats apart, ldws a
// multiple of 4, so every load is a 16-byte float4 (the up to three pad columns
// after N are read but never stored). Each thread issues kReduceBatch loads
// before adding any of them, so a launch keeps the whole workspace in flight:
// the partial rows were just written and sit in L2, and the kernel is bound by
// latency, not bandwidth (ncu at 456 partial rows of 4096: 3.8 us, against
// 4.5 us for 32-column tiles split over 4-CTA clusters; an empty kernel takes
// 1.8 us). The row sums are combined in a fixed tree: in row order within a
// thread, a butterfly over the 16 row lanes of a warp, then the warps in
// order through shared memory; the result is rounded once into the I/O dtype.
// The order depends only on (units, N), so dgamma is bitwise reproducible.
// units == 0 (no rows) writes zeros. blockIdx.y = 1 sums the second plane
// (LayerNorm's dbeta partials) into out1.
constexpr int kReduceBatch = 8;
constexpr int kReduceLanes = 2;  // float4 lanes per row: 8 columns
// `queue` (may be null): the row pool's queue word, closed here once the row
// kernel has finished (see kPoolClosed in pool.h).
template <int DT, int WARPS>
__global__ void __launch_bounds__(32 * WARPS) dgamma_reduce_kernel(const float* ws, int64_t units, int N,
                                                                  int64_t ldws, void* out0, void* out1,
                                                                  unsigned long long* queue) {
    using E = Elem<DT>;
    constexpr int kReduceRows = 32 * WARPS / kReduceLanes;  // row lanes per block
    __shared__ float4 part[WARPS][kReduceLanes];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cq = lane % kReduceLanes;
    const int ry = warp * (32 / kReduceLanes) + lane / kReduceLanes;
    const int col = blockIdx.x * (4 * kReduceLanes) + cq * 4;
    void* dgamma = blockIdx.y == 0 ? out0 : out1;
    if (blockIdx.y != 0) ws += units * ldws;
    griddep_wait();  // the partial sums come from the row kernel just before
    if (queue && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *queue = kPoolClosed;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < N) {
        for (int64_t base = ry; base < units; base += kReduceRows * kReduceBatch) {
            float4 v[kReduceBatch];
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i) {
                const int64_t p = base + kReduceRows * i;
                v[i] = p < units ? __ldcg(reinterpret_cast<const float4*>(ws + p * ldws + col))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < kReduceBatch; ++i) {
                if (base + kReduceRows * i < units) {
                    s.x += v[i].x; s.y += v[i].y; s.z += v[i].z; s.w += v[i].w;
                }
            }
        }
    }
    // the 16 row lanes of this warp
#pragma unroll
    for (int o = kReduceLanes; o < 32; o <<= 1) {
        s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
        s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
        s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
        s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
    }
    if (lane < kReduceLanes) part[warp][lane] = s;
    __syncthreads();
    if (threadIdx.x < kReduceLanes) {
        float4 t = part[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < WARPS; ++w) {
            const float4 u = part[w][threadIdx.x];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const int c = blockIdx.x * (4 * kReduceLanes) + 4 * threadIdx.x;
        if (c < N) E::st(dgamma, c, t.x);
        if (c + 1 < N) E::st(dgamma, c + 1, t.y);
        if (c + 2 < N) E::st(dgamma, c + 2, t.z);
        if (c + 3 < N) E::st(dgamma, c + 3, t.w);
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool OFF, bool CL>
static const void* bwd_tma_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&bwd_tma_kernel<DT, 1, OFF, CL>);
    case 2: return reinterpret_cast<const void*>(&bwd_tma_kernel<DT, 2, OFF, CL>);
    case 4: return reinterpret_cast<const void*>(&bwd_tma_kernel<DT, 4, OFF, CL>);
    case 8: return reinterpret_cast<const void*>(&bwd_tma_kernel<DT, 8, OFF, CL>);
    default: return nullptr;
    }
}
template <int DT, bool OFF>
static const void* bwd_pool_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&bwd_pool_kernel<DT, 1, OFF>);
    case 2: return reinterpret_cast<const void*>(&bwd_pool_kernel<DT, 2, OFF>);
    case 4: return reinterpret_cast<const void*>(&bwd_pool_kernel<DT, 4, OFF>);
    default: return nullptr;
    }
}
template <int DT, bool OFF>
static const void* bwd_tma_for(int vpt, int cluster, bool pool) {
    if (pool) return bwd_pool_vpt<DT, OFF>(vpt);
    return cluster > 1 ? bwd_tma_vpt<DT, OFF, true>(vpt) : bwd_tma_vpt<DT, OFF, false>(vpt);
}
template <int DT, bool OFF>
static const void* bwd_scalar_for() {
    return reinterpret_cast<const void*>(&bwd_scalar_kernel<DT, OFF>);
}
template <bool OFF>
static const void* bwd_pick(const Plan& p) {
    const bool tma = p.path == kPathTma;
    const bool pool = p.pool.head > 0 && p.cluster == 1;
    switch (p.dtype) {
    case kF32: return tma ? bwd_tma_for<kF32, OFF>(p.per_thread, p.cluster, pool) : bwd_scalar_for<kF32, OFF>();
    case kF16: return tma ? bwd_tma_for<kF16, OFF>(p.per_thread, p.cluster, pool) : bwd_scalar_for<kF16, OFF>();
    case kBF16: return tma ? bwd_tma_for<kBF16, OFF>(p.per_thread, p.cluster, pool) : bwd_scalar_for<kBF16, OFF>();
    default: return nullptr;
    }
}

const void* bwd_kernel(const Plan& p) {
    if (p.path == kPathLanes) return lanes_kernel(1, p);
    if (p.path == kPathRowVec) return rowvec_kernel(1, p);
    if (p.path == kPathRagged) return ragged_kernel(1, p);
    return p.offset ? bwd_pick<true>(p) : bwd_pick<false>(p);
}

template <int WARPS>
static const void* dgamma_reduce_for(int dtype) {
    switch (dtype) {
    case kF32: return reinterpret_cast<const void*>(&dgamma_reduce_kernel<kF32, WARPS>);
    case kF16: return reinterpret_cast<const void*>(&dgamma_reduce_kernel<kF16, WARPS>);
    case kBF16: return reinterpret_cast<const void*>(&dgamma_reduce_kernel<kBF16, WARPS>);
    default: return nullptr;
    }
}

// Warps per block of the column reduce: 16 (256 row lanes) above 1024 partial
// rows, so that one batch of kReduceBatch loads per lane still covers them.
int dgamma_reduce_warps(int64_t units) { return units > 1024 ? 16 : 8; }

const void* dgamma_reduce_kernel_ptr(int dtype, int64_t units) {
    return dgamma_reduce_warps(units) == 16 ? dgamma_reduce_for<16>(dtype) : dgamma_reduce_for<8>(dtype);
}


cudaError_t launch_rows(const void* k, const Plan& p, const RowArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.units * p.cluster), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads + p.extra_threads), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    if (p.cluster > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
    RowArgs args = a;
    void* params[] = {&args};
    return cudaLaunchKernelExC(&cfg, k, params);
}

cudaError_t launch_dgamma_reduce(int dtype, const float* ws, int64_t units, int N, int64_t ldws, void* dgamma,
                                 cudaStream_t s, void* dbeta, unsigned long long* queue) {
    const void* k = dgamma_reduce_kernel_ptr(dtype, units);
    if (!k) return cudaErrorInvalidDeviceFunction;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + 4 * kReduceLanes - 1) / (4 * kReduceLanes)), dbeta ? 2u : 1u, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * dgamma_reduce_warps(units)), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* params[] = {const_cast<float**>(&ws), &units, &N, &ldws, &dgamma, &dbeta, &queue};
    return cudaLaunchKernelExC(&cfg, k, params);
}

}  // namespace rmsnorm
