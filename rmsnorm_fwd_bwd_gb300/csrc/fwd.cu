// fwd.cu -- RMSNorm forward kernels.
//
// Computes, per row (page "Check an AI model calculation before accelerating
// it", section "Problem and reference formula"; offset variant from the
// torchtitan numerics page):
//     r = 1 / sqrt(sum_j(x_j^2) / N + eps);  y = (x * r) * gamma   or   ((1 + w) * x) * r
// with x widened to fp32 at load ("Why convert before reducing?") and the mean
// taken over the logical N, never over a padded width ("N and BLOCK: two sizes
// you must never confuse").
//
// Kernels:
//  * fwd_tma_kernel: persistent; each cluster of C CTAs owns rows cid, cid+K, ...
//    and CTA c of the cluster owns the column slice [c*N/C, (c+1)*N/C). A ring
//    of `stages` shared-memory buffers is filled by TMA bulk copies
//    (cp.async.bulk, one per row slice, completion on an mbarrier), so many rows
//    are in flight per SM without holding them in registers. The sum of squares
//    is reduced warp -> CTA (shared memory) -> cluster (distributed shared
//    memory) with one barrier per row; every CTA then forms the same total in the
//    same order. Output vectors go straight from registers to HBM with 16-byte
//    coalesced stores.
//  * fwd_pool_kernel: the same ring without clusters, with the row pool of
//    pool.h (a fixed head of rows per CTA, then segments of rows from a queue)
//    and a producer warp per CTA that keeps the ring full;
//  * fwd_scalar_kernel: any N and any element alignment; one CTA per row,
//    element-strided scalar loads that stay coalesced across a warp, two passes
//    over the row (the second one is served by L1/L2), few registers so that
//    many rows are in flight per SM.
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

// Minimum resident 256-thread blocks for __launch_bounds__ (0: none). The
// 64-element instances (2-byte types, 8 vectors per thread: the split-row plans,
// 128-thread blocks) are held to 128 registers, four blocks per SM.
template <int DT, int VPT> struct FwdTmaMinBlocks { static constexpr int value = Elem<DT>::kVec * VPT >= 64 ? 2 : 0; };

template <int DT, int VPT, bool OFFSET, bool CLUSTER>
__global__ void __launch_bounds__(kTmaMaxThreads, (FwdTmaMinBlocks<DT, VPT>::value)) fwd_tma_kernel(const RowArgs a) {
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

    const int ns = a.N / static_cast<int>(csize);  // slice width (elements)
    const int nvec = ns / VEC;                       // 16-byte vectors per slice
    const uint32_t slice_bytes = static_cast<uint32_t>(ns) * E::kBytes;
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    const int S = a.stages;

    // shared memory: ring | mbarriers | warp partials [2][32] | abort flag
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * slice_bytes);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;
    const char* xsl = static_cast<const char*>(a.x) + static_cast<size_t>(crank) * slice_bytes;
    char* ysl = static_cast<char*>(a.y) + static_cast<size_t>(crank) * slice_bytes;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_wait();  // inputs may come from the previous kernel on the stream
    // the first rows' copies go out before the per-column set-up below, so the
    // ring fills while gamma is being loaded
    const uint64_t pol = l2_evict_first_policy();
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) {
            const uint32_t bar = smem_u32(&full[j]);
            mbar_arrive_expect_tx(bar, slice_bytes);
            bulk_g2s_in(smem_u32(ring + j * slice_bytes), xsl + static_cast<size_t>(cid + j * ncl) * x_pitch,
                        slice_bytes, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
        }
    }

    // gamma slice widened to fp32 once (offset variant: 1 + w), kept in registers;
    // at 64 elements per thread (2-byte types, 8 vectors) x and gamma stay as raw
    // 16-byte words instead and are widened where used, which halves their
    // registers and lets more blocks share an SM
    constexpr bool PACK = VEC * VPT >= 64;
    float gf[PACK ? 1 : VPT][VEC];
    uint4 gr[PACK ? VPT : 1];
    {
        const uint4* gs = reinterpret_cast<const uint4*>(
            static_cast<const char*>(a.gamma) + static_cast<size_t>(crank) * slice_bytes);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            const uint4 raw = idx < nvec ? __ldg(gs + idx) : make_uint4(0, 0, 0, 0);
            if constexpr (PACK) {
                gr[v] = raw;
            } else {
                E::unpack(raw, gf[v]);
                if (OFFSET) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) gf[v][e] = 1.0f + gf[v][e];
                }
            }
        }
    }

    __syncthreads();
    if (CLUSTER) cluster_sync();  // peers' shared memory is live before any DSMEM read

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = cid + j * ncl;
        const unsigned char* st = ring + static_cast<size_t>(s) * slice_bytes;

        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        // x slice widened to fp32 once (or kept raw, see PACK); sum of squares on the way
        float xf[PACK ? 1 : VPT][VEC];
        uint4 xr[PACK ? VPT : 1];
        // two sums of squares, even and odd elements: the two lanes of one packed
        // f32x2 register, except in the 64-element instances (PACK), where the
        // packed form measured slower (fp16 16384x16384 forward: 175.9 us scalar,
        // 177.8 packed)
        uint64_t ss = f2_pack(0.f, 0.f);
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            const uint4 raw = idx < nvec ? *reinterpret_cast<const uint4*>(st + idx * 16) : make_uint4(0, 0, 0, 0);
            float* xv = xf[PACK ? 0 : v];
            if constexpr (PACK) xr[v] = raw;
            E::unpack(raw, *reinterpret_cast<float(*)[VEC]>(xv));
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                if constexpr (PACK) {
                    ss0 = fmaf(xv[e], xv[e], ss0);
                    ss1 = fmaf(xv[e + 1], xv[e + 1], ss1);
                } else {
                    const uint64_t x2 = f2_pack(xv[e], xv[e + 1]);
                    ss = f2_fma(x2, x2, ss);
                }
            }
        }
        if constexpr (!PACK) f2_unpack(ss, ss0, ss1);
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(ss0 + ss1);
        if (lane == 0) redb[warp] = wsum;
        // every thread has its slice in registers after this barrier: the stage can refill
        if (CLUSTER) cluster_sync(); else __syncthreads();
        if (!aborted && *abort_flag) {
            aborted = true;
            abort_row = j;
        }

        if (tid == 0 && !aborted && j + S < nrows) {
            fence_proxy_async_smem();
            const uint32_t bar = smem_u32(&full[s]);
            mbar_arrive_expect_tx(bar, slice_bytes);
            bulk_g2s_in(smem_u32(st), xsl + static_cast<size_t>(row + S * ncl) * x_pitch, slice_bytes, bar, pol,
                        a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
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
        const float ms = t / static_cast<float>(a.N);
        const float r = 1.0f / sqrtf(ms + a.eps);

        if (!aborted) {
            if (tid == 0 && crank == 0) a.rstd_out[row] = r;
            char* yrow = ysl + static_cast<size_t>(row) * y_pitch;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nt + tid;
                if (idx < nvec) {
                    float o[VEC];
                    if constexpr (PACK) {
                        float xv[VEC], gv[VEC];
                        // empty asm statements mark the raw words as changed, so the
                        // compiler neither hoists gamma's widening out of the row
                        // loop nor keeps x's widened values from the sum of squares
                        // live across the barrier (64 registers each)
                        uint4 gw = gr[v], xw = xr[v];
                        asm volatile("" : "+r"(gw.x), "+r"(gw.y), "+r"(gw.z), "+r"(gw.w));
                        asm volatile("" : "+r"(xw.x), "+r"(xw.y), "+r"(xw.z), "+r"(xw.w));
                        E::unpack(xw, xv);
                        E::unpack(gw, gv);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const float g = OFFSET ? 1.0f + gv[e] : gv[e];
                            o[e] = OFFSET ? (g * xv[e]) * r : (xv[e] * r) * g;
                        }
                    } else {
                        scale_pairs<VEC, OFFSET>(xf[v], gf[v], false, r, o);
                    }
                    stg128(yrow + idx * 16, E::pack(o));
                }
            }
        }
    }
    griddep_launch_dependents();
    if (CLUSTER) cluster_sync();  // no CTA leaves while a peer may read its shared memory
    if (aborted && tid == 0) {
        // copies issued for rows abort_row .. abort_row+S-1 may still be in flight
        const int64_t end = abort_row + S < nrows ? abort_row + S : nrows;
        for (int64_t j = abort_row; j < end; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), static_cast<uint32_t>((j / S) & 1), a.err, 1u << 16);
    }
}

// The forward's queue words: one per call slot, in the library's own device
// memory (the forward has no workspace). A call's CTA 0 opens its slot by storing
// {ticket, 0}; a take whose fetch-and-add finds another ticket there (another call
// given the same slot and running at the same time, or a take that came before
// CTA 0's store) cannot trust the count, and that CTA then runs every segment of
// the queue itself: rows written twice get the same values, so the result stays
// right, only slower. Cleared at load; read and written only by forward pool
// kernels.
__device__ unsigned long long g_fwd_queue[kFwdQueueSlots];

// Forward row kernel with the row pool of pool.h (no clusters), formulas as in
// fwd_tma_kernel. CTA b takes rows b + j * G, j < a.pool.head, then segments of
// consecutive rows from the call's queue word. a.threads consumer threads plus one
// producer warp: the producer's lane 0 runs the TMA ring ahead of the consumers
// (`full` barriers for the copies, `empty` barriers, one arrival per consumer
// warp, before a stage is refilled), decides each stage's row and records it in
// shared memory; a stage with no row (queue empty) ends both loops. The
// consumers sync only on a named barrier (the row's sum of squares).
// a.pool_solo (tuning) makes every CTA run every segment.
template <int DT, int VPT, bool OFFSET>
__global__ void __launch_bounds__(kTmaMaxThreads + 32) fwd_pool_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int64_t stage_row[kPoolMaxStages];
    __shared__ uint64_t empty[kPoolMaxStages];

    const int tid = threadIdx.x;
    const int nc = blockDim.x - 32;  // consumer threads
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int ncw = nc >> 5;
    const int64_t G = gridDim.x;
    const int nvec = a.N / VEC;
    const uint32_t row_bytes = static_cast<uint32_t>(a.N) * E::kBytes;
    const int S = a.stages;

    // shared memory: ring | full barriers | warp partials [2][32] | abort flag
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * row_bytes);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
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
        const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
        int64_t heads = 0, seg_row = 0, seg_end = 0, seg_id = -1;
        bool solo = a.pool_solo != 0, done = false;
        unsigned long long pend = 0;
        bool pend_on = false;
        auto take_ahead = [&]() {
            if (!pend_on && !solo) {
                pend = atomicAdd(a.queue, 1ull);
                pend_on = true;
            }
        };
        int64_t issued = 0;
        bool aborted = false;
        for (;; ++issued) {
            const int s = static_cast<int>(issued % S);
            const int64_t round = issued / S;
            if (round > 0) {
                bool ok = false;
#pragma unroll 1
                for (uint32_t i = 0; i < kWaitPollLimit && !ok; ++i) {
                    ok = mbar_try_wait(smem_u32(&empty[s]), static_cast<uint32_t>((round - 1) & 1));
                    if (!ok && *abort_flag) break;
                }
                if (!ok) {
                    if (!*abort_flag) atomicOr(a.err, kDevErrWaitTimeout);
                    aborted = true;
                    break;
                }
            }
            int64_t row = -1;
            if (heads < a.pool.head) {
                row = static_cast<int64_t>(blockIdx.x) + heads * G;
                ++heads;
                if (a.pool.head - heads <= kPoolTakeAhead) take_ahead();
            } else if (!done) {
                if (seg_row >= seg_end) {
                    int64_t k;
                    if (solo) {
                        k = seg_id + 1;
                    } else {
                        take_ahead();
                        pend_on = false;
                        if ((pend >> 32) == ticket) {
                            k = static_cast<int64_t>(pend & 0xffffffffull);
                        } else {
                            solo = true;  // the count is not this call's: run every segment
                            k = 0;
                        }
                    }
                    if (k < a.pool.nseg) {
                        pool_segment(a.pool, k, seg_row, seg_end);
                        seg_id = k;
                    } else {
                        done = true;
                    }
                }
                if (!done) {
                    row = seg_row++;
                    if (seg_end - seg_row <= kPoolTakeAhead) take_ahead();
                }
            }
            stage_row[s] = row;
            const uint32_t bar = smem_u32(&full[s]);
            if (row < 0) {
                mbar_arrive(bar);
                break;
            }
            mbar_arrive_expect_tx(bar, row_bytes);
            bulk_g2s_in(smem_u32(ring + static_cast<size_t>(s) * row_bytes), xb + static_cast<size_t>(row) * x_pitch,
                        row_bytes, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
            if (issued == 0 && blockIdx.x == 0) atomicExch(a.queue, static_cast<unsigned long long>(ticket) << 32);
        }
        if (aborted) {
            for (int64_t i = issued - S < 0 ? 0 : issued - S; i < issued; ++i)
                if (stage_row[i % S] >= 0)
                    mbar_wait_bounded(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), a.err,
                                      1u << 16);
        }
        return;
    }

    // ---------------- consumers ----------------
    float gf[VPT][VEC];
    {
        const uint4* gs = reinterpret_cast<const uint4*>(a.gamma);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nc + tid;
            const uint4 raw = idx < nvec ? __ldg(gs + idx) : make_uint4(0, 0, 0, 0);
            E::unpack(raw, gf[v]);
            if (OFFSET) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) gf[v][e] = 1.0f + gf[v][e];
            }
        }
    }
    char* yb = static_cast<char*>(a.y);
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0;; ++j) {
        if (!mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;
        const int64_t row = stage_row[s];
        if (row < 0) break;  // the queue is empty (every consumer reads the same stage)
        const unsigned char* st = ring + static_cast<size_t>(s) * row_bytes;
        float xf[VPT][VEC];
        uint64_t ss = f2_pack(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nc + tid;
            const uint4 raw = idx < nvec ? *reinterpret_cast<const uint4*>(st + idx * 16) : make_uint4(0, 0, 0, 0);
            E::unpack(raw, xf[v]);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const uint64_t x2 = f2_pack(xf[v][e], xf[v][e + 1]);
                ss = f2_fma(x2, x2, ss);
            }
        }
        // this warp is done with the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        float ss0, ss1;
        f2_unpack(ss, ss0, ss1);
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(ss0 + ss1);
        if (lane == 0) redb[warp] = wsum;
        named_barrier_sync(1, nc);
        if (*abort_flag) break;  // every consumer reads the flag after the same barrier
        float t = lane < ncw ? redb[lane] : 0.f;
        t = warp_allsum(t);
        const float ms = t / static_cast<float>(a.N);
        const float r = 1.0f / sqrtf(ms + a.eps);
        if (tid == 0) a.rstd_out[row] = r;
        char* yrow = yb + static_cast<size_t>(row) * y_pitch;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nc + tid;
            if (idx < nvec) {
                float o[VEC];
                scale_pairs<VEC, OFFSET>(xf[v], gf[v], false, r, o);
                stg128(yrow + idx * 16, E::pack(o));
            }
        }
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
    griddep_launch_dependents();
}

template <int DT, bool OFFSET>
__global__ void __launch_bounds__(kScalarThreads) fwd_scalar_kernel(const RowArgs a) {
    using E = Elem<DT>;
    __shared__ float red[2][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    griddep_wait();

    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t base = row * a.ldx;
        const int64_t ybase = row * a.ldy;
        // pass 1: sum of squares, four independent loads in flight per thread
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int col = tid;
        for (; col + 3 * nt < N; col += 4 * nt) {
            const float v0 = E::ld(a.x, base + col);
            const float v1 = E::ld(a.x, base + col + nt);
            const float v2 = E::ld(a.x, base + col + 2 * nt);
            const float v3 = E::ld(a.x, base + col + 3 * nt);
            s0 = fmaf(v0, v0, s0);
            s1 = fmaf(v1, v1, s1);
            s2 = fmaf(v2, v2, s2);
            s3 = fmaf(v3, v3, s3);
        }
        for (; col < N; col += nt) {
            const float v = E::ld(a.x, base + col);
            s0 = fmaf(v, v, s0);
        }
        const float ws = warp_allsum((s0 + s1) + (s2 + s3));
        if (lane == 0) red[parity][warp] = ws;
        __syncthreads();
        float t = lane < nwarps ? red[parity][lane] : 0.f;
        t = warp_allsum(t);
        const float r = 1.0f / sqrtf(t / static_cast<float>(N) + a.eps);
        if (tid == 0) a.rstd_out[row] = r;
        // pass 2: the row again (now in L1/L2), gamma, output
#pragma unroll 4
        for (int c = tid; c < N; c += nt) {
            const float xv = E::ld(a.x, base + c);
            const float w = E::ld(a.gamma, c);
            const float g = OFFSET ? 1.0f + w : w;
            E::st(a.y, ybase + c, OFFSET ? (g * xv) * r : (xv * r) * g);
        }
    }
    griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool OFF, bool CL>
static const void* fwd_tma_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&fwd_tma_kernel<DT, 1, OFF, CL>);
    case 2: return reinterpret_cast<const void*>(&fwd_tma_kernel<DT, 2, OFF, CL>);
    case 4: return reinterpret_cast<const void*>(&fwd_tma_kernel<DT, 4, OFF, CL>);
    case 8: return reinterpret_cast<const void*>(&fwd_tma_kernel<DT, 8, OFF, CL>);
    default: return nullptr;
    }
}
template <int DT, bool OFF>
static const void* fwd_pool_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&fwd_pool_kernel<DT, 1, OFF>);
    case 2: return reinterpret_cast<const void*>(&fwd_pool_kernel<DT, 2, OFF>);
    case 4: return reinterpret_cast<const void*>(&fwd_pool_kernel<DT, 4, OFF>);
    default: return nullptr;
    }
}
template <int DT, bool OFF>
static const void* fwd_tma_for(int vpt, int cluster, bool pool) {
    if (pool) return fwd_pool_vpt<DT, OFF>(vpt);
    return cluster > 1 ? fwd_tma_vpt<DT, OFF, true>(vpt) : fwd_tma_vpt<DT, OFF, false>(vpt);
}
template <int DT, bool OFF>
static const void* fwd_scalar_for() {
    return reinterpret_cast<const void*>(&fwd_scalar_kernel<DT, OFF>);
}
template <bool OFF>
static const void* fwd_pick(const Plan& p) {
    const bool tma = p.path == kPathTma;
    const bool pool = p.pool.head > 0 && p.cluster == 1;
    switch (p.dtype) {
    case kF32: return tma ? fwd_tma_for<kF32, OFF>(p.per_thread, p.cluster, pool) : fwd_scalar_for<kF32, OFF>();
    case kF16: return tma ? fwd_tma_for<kF16, OFF>(p.per_thread, p.cluster, pool) : fwd_scalar_for<kF16, OFF>();
    case kBF16: return tma ? fwd_tma_for<kBF16, OFF>(p.per_thread, p.cluster, pool) : fwd_scalar_for<kBF16, OFF>();
    default: return nullptr;
    }
}

unsigned long long* fwd_queue_word(unsigned slot) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_queue) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<unsigned long long*>(p) + slot % kFwdQueueSlots;
}

const void* fwd_kernel(const Plan& p) {
    if (p.path == kPathLanes) return lanes_kernel(0, p);
    if (p.path == kPathRowVec) return rowvec_kernel(0, p);
    if (p.path == kPathRagged) return ragged_kernel(0, p);
    return p.offset ? fwd_pick<true>(p) : fwd_pick<false>(p);
}

}  // namespace rmsnorm
