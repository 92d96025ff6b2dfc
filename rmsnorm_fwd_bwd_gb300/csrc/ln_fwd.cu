// ln_fwd.cu -- LayerNorm forward kernels.
//
// Per row (page "torch.compile performance leap: optimizing LayerNorm and
// RMSNorm kernels", section 1.1: mean and variance of the row, learned weight
// gamma and bias beta; the page prints no formula, so this is the standard one):
//     mu = sum_j x_j / N;  var = sum_j (x_j - mu)^2 / N;  r = 1 / sqrt(var + eps)
//     y = ((x - mu) * r) * gamma + beta
// mu and r are saved (fp32) for the backward when their pointers are not null
// (section 1.4: mean and variance are stored only when a backward will need them).
//
// Two kernels, on the same machinery as the RMSNorm forward:
//  * ln_fwd_tma_kernel: persistent, TMA bulk-copy ring, rows split over a
//    thread-block cluster when they are wide. The mean and the variance take
//    ONE barrier per row. Each warp forms, from registers, the mean of its
//    elements (a butterfly sum) and then the sum of squared deviations about
//    that mean (a second butterfly sum): a two-pass variance within the warp.
//    The per-warp triples (count n_w, mean m_w, deviations q_w) of the CTA, or
//    of every CTA of the cluster through distributed shared memory, are then
//    combined by the parallel-axis identity
//        mu = sum_w n_w m_w / N,   q = sum_w (q_w + n_w (m_w - mu)^2)
//    with two more butterfly sums, whose every term is non-negative. No
//    one-pass sum-of-squares formula: rows with a large mean keep their
//    accuracy. Butterfly sums leave the same bits in every lane, so every
//    thread of every CTA of the row uses the same mu and r.
//  * ln_fwd_scalar_kernel: any N and element alignment (rows too wide for the
//    row-vector kernels of ln_rowvec.cu), one CTA per row, three
//    passes over the row (sum; squared deviations; output), the later ones
//    served by L1/L2.
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

template <int DT, int VPT, bool CLUSTER>
__global__ void __launch_bounds__(kTmaMaxThreads) ln_fwd_tma_kernel(const RowArgs a) {
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
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    const int S = a.stages;

    // shared memory: ring | mbarriers | warp partials n, m, q [2][32] each | abort flag
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * slice_bytes);
    float* red_n = reinterpret_cast<float*>(full + S);
    float* red_m = red_n + 64;
    float* red_q = red_n + 128;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red_n + 192);

    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;
    const size_t slice_off = static_cast<size_t>(crank) * slice_bytes;
    const char* xsl = static_cast<const char*>(a.x) + slice_off;
    char* ysl = static_cast<char*>(a.y) + slice_off;

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

    // gamma and beta slices widened to fp32 once, kept in registers
    float gf[VPT][VEC], bf[VPT][VEC];
    {
        const uint4* gs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.gamma) + slice_off);
        const uint4* bs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.beta) + slice_off);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            E::unpack(idx < nvec ? __ldg(gs + idx) : make_uint4(0, 0, 0, 0), gf[v]);
            E::unpack(idx < nvec ? __ldg(bs + idx) : make_uint4(0, 0, 0, 0), bf[v]);
        }
    }
    // elements this warp owns in every row (a multiple of VEC)
    int mine = 0;
#pragma unroll
    for (int v = 0; v < VPT; ++v) mine += (v * nt + tid < nvec) ? VEC : 0;
    const float n_warp = warp_allsum(static_cast<float>(mine));

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

        // x slice widened to fp32 once; the warp's mean, then its squared deviations
        float xf[VPT][VEC];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            E::unpack(idx < nvec ? *reinterpret_cast<const uint4*>(st + idx * 16) : make_uint4(0, 0, 0, 0),
                      xf[v]);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 += xf[v][e];
                s1 += xf[v][e + 1];
            }
        }
        // a true division: equal elements give back their value exactly
        const float m_warp = n_warp > 0.f ? warp_allsum(s0 + s1) / n_warp : 0.f;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            if (v * nt + tid < nvec) {
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    const float d0 = xf[v][e] - m_warp, d1 = xf[v][e + 1] - m_warp;
                    q0 = fmaf(d0, d0, q0);
                    q1 = fmaf(d1, d1, q1);
                }
            }
        }
        const float q_warp = warp_allsum(q0 + q1);
        const int b = static_cast<int>(j & 1) * 32;
        if (lane == 0) {
            red_n[b + warp] = n_warp;
            red_m[b + warp] = m_warp;
            red_q[b + warp] = q_warp;
        }
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

        // lane l holds warp (l mod nwarps) of CTA (l / nwarps); empty lanes hold n = 0
        float tn = 0.f, tm = 0.f, tq = 0.f;
        if (!CLUSTER) {
            if (lane < nwarps) {
                tn = red_n[b + lane];
                tm = red_m[b + lane];
                tq = red_q[b + lane];
            }
        } else if (lane < nwarps * static_cast<int>(csize)) {
            const uint32_t rk = static_cast<uint32_t>(lane / nwarps);
            const int w = lane % nwarps;
            tn = dsmem_ld_f32(dsmem_map(smem_u32(red_n + b + w), rk));
            tm = dsmem_ld_f32(dsmem_map(smem_u32(red_m + b + w), rk));
            tq = dsmem_ld_f32(dsmem_map(smem_u32(red_q + b + w), rk));
        }
        const float mu = warp_allsum(tn * tm) / static_cast<float>(a.N);
        const float dm = tm - mu;
        const float var = warp_allsum(fmaf(tn * dm, dm, tq)) / static_cast<float>(a.N);
        const float r = 1.0f / sqrtf(var + a.eps);

        if (!aborted) {
            if (tid == 0 && crank == 0) {
                if (a.mean_out) a.mean_out[row] = mu;
                if (a.rstd_out) a.rstd_out[row] = r;
            }
            char* yrow = ysl + static_cast<size_t>(row) * y_pitch;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nt + tid;
                if (idx < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf((xf[v][e] - mu) * r, gf[v][e], bf[v][e]);
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

// Block-wide sum of one value per thread; every thread gets the same bits.
// `red` holds 32 floats; callers alternate buffers between consecutive calls.
__device__ __forceinline__ float block_allsum(float v, float* red) {
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    v = warp_allsum(v);
    if (lane == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = lane < nwarps ? red[lane] : 0.f;
    return warp_allsum(t);
}

template <int DT>
__global__ void __launch_bounds__(kScalarThreads) ln_fwd_scalar_kernel(const RowArgs a) {
    using E = Elem<DT>;
    // two buffers: the sum of a row and its squared deviations. A thread writes
    // the first buffer of the next row only after the second barrier of this
    // row, which every thread passes after reading the first one.
    __shared__ float red[2][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int N = a.N;
    griddep_wait();

    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * a.ldx;
        const int64_t ybase = row * a.ldy;
        float s0 = 0.f, s1 = 0.f;
        int col = tid;
        for (; col + nt < N; col += 2 * nt) {
            s0 += E::ld(a.x, base + col);
            s1 += E::ld(a.x, base + col + nt);
        }
        if (col < N) s0 += E::ld(a.x, base + col);
        const float mu = block_allsum(s0 + s1, red[0]) / static_cast<float>(N);
        float q0 = 0.f, q1 = 0.f;
        col = tid;
        for (; col + nt < N; col += 2 * nt) {
            const float d0 = E::ld(a.x, base + col) - mu;
            const float d1 = E::ld(a.x, base + col + nt) - mu;
            q0 = fmaf(d0, d0, q0);
            q1 = fmaf(d1, d1, q1);
        }
        if (col < N) {
            const float d0 = E::ld(a.x, base + col) - mu;
            q0 = fmaf(d0, d0, q0);
        }
        const float var = block_allsum(q0 + q1, red[1]) / static_cast<float>(N);
        const float r = 1.0f / sqrtf(var + a.eps);
        if (tid == 0) {
            if (a.mean_out) a.mean_out[row] = mu;
            if (a.rstd_out) a.rstd_out[row] = r;
        }
#pragma unroll 4
        for (int c = tid; c < N; c += nt) {
            const float xh = (E::ld(a.x, base + c) - mu) * r;
            E::st(a.y, ybase + c, fmaf(xh, E::ld(a.gamma, c), E::ld(a.beta, c)));
        }
    }
    griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool CL>
static const void* ln_fwd_tma_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&ln_fwd_tma_kernel<DT, 1, CL>);
    case 2: return reinterpret_cast<const void*>(&ln_fwd_tma_kernel<DT, 2, CL>);
    case 4: return reinterpret_cast<const void*>(&ln_fwd_tma_kernel<DT, 4, CL>);
    case 8: return reinterpret_cast<const void*>(&ln_fwd_tma_kernel<DT, 8, CL>);
    default: return nullptr;
    }
}
template <int DT>
static const void* ln_fwd_for(const Plan& p) {
    if (p.path == kPathScalar) return reinterpret_cast<const void*>(&ln_fwd_scalar_kernel<DT>);
    if (p.path != kPathTma) return nullptr;
    return p.cluster > 1 ? ln_fwd_tma_vpt<DT, true>(p.per_thread) : ln_fwd_tma_vpt<DT, false>(p.per_thread);
}

const void* ln_fwd_kernel(const Plan& p) {
    if (p.path == kPathLanes) return lanes_kernel(2, p);
    if (p.path == kPathRowVec) return ln_rowvec_kernel(2, p);
    if (p.path == kPathRagged) return ln_ragged_kernel(2, p);
    switch (p.dtype) {
    case kF32: return ln_fwd_for<kF32>(p);
    case kF16: return ln_fwd_for<kF16>(p);
    case kBF16: return ln_fwd_for<kBF16>(p);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
