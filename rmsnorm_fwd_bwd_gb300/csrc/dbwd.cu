// dbwd.cu -- RMSNorm double backward: the gradient of the backward pass.
//
// The backward maps (dy, x, g) to (dx, dgamma) with g = gamma or 1 + w. For
// cotangents ddx of dx and ddg of dgamma, differentiating the backward (r
// depends on x through dr/dx_j = -r^3 x_j / N) gives, per row, with
//     u = dy*g,  c = mean(u*x),  A = mean(ddx*x),  B = mean(ddx*u),
//     D = mean(ddg*dy*x),  e = ddx - r^2*x*A:
//     d_dy = g*r*e + r*x*ddg
//     d_x  = r*ddg*dy - r^3*(c*ddx + u*A + x*(B + D)) + 3*r^5*c*A*x
//     d_g  = sum over rows of r*dy*e
// (the page "Check an AI model calculation before accelerating it", section
// "Adapting the kernel and moving to production", lists double backward among
// the extensions it did not validate). ddg may be absent (zero).
//
// Two kernels, on the backward's machinery:
//  * dbwd_tma_kernel: persistent; one ring stage holds the x, dy and ddx slices
//    of a row (TMA bulk copies); g and ddg sit in shared memory as fp32 float4
//    planes; the four row sums take one barrier (CTA or cluster); d_dy and d_x
//    leave as 16-byte stores; fp32 d_g accumulators per thread over the block's
//    rows become one row of the workspace, summed by the fixed-order column
//    reduce.
//  * dbwd_scalar_kernel: any N and element alignment; one CTA per row, two
//    passes over the row (the second served by L1/L2), d_g accumulators in
//    shared memory.
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

// Block-size bound: up to kDbwdMaxThreads for the single-CTA plans of at most two
// vectors per thread (at most 116 registers under it, so the 256-thread plans
// keep two blocks per SM), kTmaMaxThreads otherwise. One 512-thread block per
// row replaces a two-CTA cluster and its cluster barrier per row: fp16 offset
// 16384x8192 285.8 -> 228.7 us.
template <int VPT, bool CLUSTER> struct DbwdTmaThreads {
    static constexpr int value = (!CLUSTER && VPT <= 2) ? kDbwdMaxThreads : kTmaMaxThreads;
};

template <int DT, int VPT, bool OFFSET, bool CLUSTER>
__global__ void __launch_bounds__(DbwdTmaThreads<VPT, CLUSTER>::value) dbwd_tma_kernel(const RowArgs a) {
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
    const uint32_t stage_bytes = 3 * slice_bytes;  // x, dy, ddx slices
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
    const size_t t_pitch = static_cast<size_t>(a.ldddx) * E::kBytes;
    const size_t odx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const size_t ody_pitch = static_cast<size_t>(a.ldd_dy) * E::kBytes;
    const int S = a.stages;

    // shared memory: ring | g slice fp32 | ddg slice fp32 | mbarriers | partials [2][4][32] | abort flag
    unsigned char* ring = smem;
    float* gsm = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * stage_bytes);
    float* qsm = gsm + ns;
    uint64_t* full = reinterpret_cast<uint64_t*>(qsm + ns);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 256);

    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;
    const size_t slice_off = static_cast<size_t>(crank) * slice_bytes;
    const char* xsl = static_cast<const char*>(a.x) + slice_off;
    const char* dysl = static_cast<const char*>(a.dy) + slice_off;
    const char* tsl = static_cast<const char*>(a.ddx) + slice_off;
    char* odx = static_cast<char*>(a.dx) + slice_off;
    char* ody = static_cast<char*>(a.d_dy) + slice_off;

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
        bulk_g2s_in(smem_u32(st + 2 * slice_bytes), tsl + r * t_pitch, slice_bytes, bar, pol,
                    a.ddx, a.M, a.ldddx, a.N, E::kBytes, a.err);
    };
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) issue(j, ring + j * stage_bytes, smem_u32(&full[j]));
    }

    // g (or 1 + w) and ddg slices widened once into shared memory as VEC/4 planes of float4
    float4* gsm4 = reinterpret_cast<float4*>(gsm);
    float4* qsm4 = reinterpret_cast<float4*>(qsm);
    {
        const uint4* gs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.gamma) + slice_off);
        const uint4* qs = a.ddg ? reinterpret_cast<const uint4*>(static_cast<const char*>(a.ddg) + slice_off)
                                : nullptr;
        for (int idx = tid; idx < nvec; idx += nt) {
            float w[VEC], q[VEC];
            E::unpack(__ldg(gs + idx), w);
            E::unpack(qs ? __ldg(qs + idx) : make_uint4(0, 0, 0, 0), q);
#pragma unroll
            for (int k = 0; k < VEC; k += 4) {
                gsm4[(k / 4) * nvec + idx] =
                    OFFSET ? make_float4(1.0f + w[k], 1.0f + w[k + 1], 1.0f + w[k + 2], 1.0f + w[k + 3])
                           : make_float4(w[k], w[k + 1], w[k + 2], w[k + 3]);
                qsm4[(k / 4) * nvec + idx] = make_float4(q[k], q[k + 1], q[k + 2], q[k + 3]);
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
    auto rstd_at = [&](int64_t jj) -> float { return jj < nrows ? __ldg(a.rstd_in + cid + jj * ncl) : 0.f; };
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

        // x, dy and ddx widened once and kept in registers; the four row sums
        float xf[VPT][VEC], df[VPT][VEC], tf[VPT][VEC];
        float pc = 0.f, pa = 0.f, pb = 0.f, pd = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            if (idx < nvec) {
                E::unpack(*reinterpret_cast<const uint4*>(st + idx * 16), xf[v]);
                E::unpack(*reinterpret_cast<const uint4*>(st + slice_bytes + idx * 16), df[v]);
                E::unpack(*reinterpret_cast<const uint4*>(st + 2 * slice_bytes + idx * 16), tf[v]);
#pragma unroll
                for (int k = 0; k < VEC; k += 4) {
                    const float4 g4 = gsm4[(k / 4) * nvec + idx];
                    const float4 q4 = qsm4[(k / 4) * nvec + idx];
                    const float g[4] = {g4.x, g4.y, g4.z, g4.w};
                    const float q[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x = xf[v][k + e], d = df[v][k + e], t = tf[v][k + e];
                        const float u = __fmul_rn(d, g[e]);
                        pc = fmaf(u, x, pc);
                        pa = fmaf(t, x, pa);
                        pb = fmaf(t, u, pb);
                        pd = fmaf(__fmul_rn(q[e], d), x, pd);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) xf[v][e] = df[v][e] = tf[v][e] = 0.f;
            }
        }
        float* redb = red + (j & 1) * 128;
        const float w0 = warp_allsum(pc), w1 = warp_allsum(pa), w2 = warp_allsum(pb), w3 = warp_allsum(pd);
        if (lane == 0) {
            redb[warp] = w0;
            redb[32 + warp] = w1;
            redb[64 + warp] = w2;
            redb[96 + warp] = w3;
        }
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

        float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
        if (!CLUSTER) {
            if (lane < nwarps) {
                t0 = redb[lane];
                t1 = redb[32 + lane];
                t2 = redb[64 + lane];
                t3 = redb[96 + lane];
            }
        } else if (lane < nwarps * static_cast<int>(csize)) {
            const uint32_t rk = static_cast<uint32_t>(lane / nwarps);
            const int w = lane % nwarps;
            t0 = dsmem_ld_f32(dsmem_map(smem_u32(redb + w), rk));
            t1 = dsmem_ld_f32(dsmem_map(smem_u32(redb + 32 + w), rk));
            t2 = dsmem_ld_f32(dsmem_map(smem_u32(redb + 64 + w), rk));
            t3 = dsmem_ld_f32(dsmem_map(smem_u32(redb + 96 + w), rk));
        }
        const float inv_n = 1.0f / static_cast<float>(a.N);
        const float c = warp_allsum(t0) * inv_n;
        const float A = warp_allsum(t1) * inv_n;
        const float bd = (warp_allsum(t2) + warp_allsum(t3)) * inv_n;  // B + D
        const float r2 = r * r;
        const float r3 = r2 * r;
        const float r2a = r2 * A;
        const float k5 = (3.0f * (r3 * r2)) * (c * A);

        if (!aborted) {
            char* odx_row = odx + static_cast<size_t>(row) * odx_pitch;
            char* ody_row = ody + static_cast<size_t>(row) * ody_pitch;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nt + tid;
                if (idx < nvec) {
                    float o_dy[VEC], o_x[VEC];
#pragma unroll
                    for (int k = 0; k < VEC; k += 4) {
                        const float4 g4 = gsm4[(k / 4) * nvec + idx];
                        const float4 q4 = qsm4[(k / 4) * nvec + idx];
                        const float g[4] = {g4.x, g4.y, g4.z, g4.w};
                        const float q[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x = xf[v][k + e], d = df[v][k + e], t = tf[v][k + e];
                            const float u = __fmul_rn(d, g[e]);
                            const float ee = fmaf(-r2a, x, t);  // ddx - r^2 x A
                            o_dy[k + e] = fmaf(g[e] * r, ee, (r * x) * q[e]);
                            const float inner = fmaf(x, bd, fmaf(c, t, u * A));
                            o_x[k + e] = fmaf(k5, x, fmaf(-r3, inner, (r * q[e]) * d));
                            acc[v][k + e] = fmaf(r * d, ee, acc[v][k + e]);
                        }
                    }
                    stg128(ody_row + idx * 16, E::pack(o_dy));
                    stg128(odx_row + idx * 16, E::pack(o_x));
                }
            }
        }
    }

    griddep_launch_dependents();
    if (!aborted) {
        float* wrow = a.ws + static_cast<size_t>(cid) * a.ldws + static_cast<size_t>(crank) * ns;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            if (idx < nvec) {
#pragma unroll
                for (int k = 0; k < VEC; k += 4)
                    *reinterpret_cast<float4*>(wrow + idx * VEC + k) =
                        make_float4(acc[v][k], acc[v][k + 1], acc[v][k + 2], acc[v][k + 3]);
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

template <int DT, bool OFFSET>
__global__ void __launch_bounds__(kScalarThreads) dbwd_scalar_kernel(const RowArgs a) {
    using E = Elem<DT>;
    extern __shared__ __align__(16) unsigned char smem[];
    float* acc = reinterpret_cast<float*>(smem);  // [N]
    __shared__ float red[2][4][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    griddep_wait();

    for (int col = tid; col < N; col += nt) acc[col] = 0.f;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t xb = row * a.ldx, db = row * a.lddy, tb = row * a.ldddx;
        const float r = __ldg(a.rstd_in + row);
        float pc = 0.f, pa = 0.f, pb = 0.f, pd = 0.f;
        for (int col = tid; col < N; col += nt) {
            const float w = E::ld(a.gamma, col);
            const float g = OFFSET ? 1.0f + w : w;
            const float q = a.ddg ? E::ld(a.ddg, col) : 0.f;
            const float x = E::ld(a.x, xb + col), d = E::ld(a.dy, db + col), t = E::ld(a.ddx, tb + col);
            const float u = __fmul_rn(d, g);
            pc = fmaf(u, x, pc);
            pa = fmaf(t, x, pa);
            pb = fmaf(t, u, pb);
            pd = fmaf(__fmul_rn(q, d), x, pd);
        }
        const float w0 = warp_allsum(pc), w1 = warp_allsum(pa), w2 = warp_allsum(pb), w3 = warp_allsum(pd);
        if (lane == 0) {
            red[parity][0][warp] = w0;
            red[parity][1][warp] = w1;
            red[parity][2][warp] = w2;
            red[parity][3][warp] = w3;
        }
        __syncthreads();
        const float inv_n = 1.0f / static_cast<float>(N);
        const float c = warp_allsum(lane < nwarps ? red[parity][0][lane] : 0.f) * inv_n;
        const float A = warp_allsum(lane < nwarps ? red[parity][1][lane] : 0.f) * inv_n;
        const float bd = (warp_allsum(lane < nwarps ? red[parity][2][lane] : 0.f) +
                          warp_allsum(lane < nwarps ? red[parity][3][lane] : 0.f)) * inv_n;
        const float r2 = r * r;
        const float r3 = r2 * r;
        const float r2a = r2 * A;
        const float k5 = (3.0f * (r3 * r2)) * (c * A);
#pragma unroll 4
        for (int col = tid; col < N; col += nt) {
            const float w = E::ld(a.gamma, col);
            const float g = OFFSET ? 1.0f + w : w;
            const float q = a.ddg ? E::ld(a.ddg, col) : 0.f;
            const float x = E::ld(a.x, xb + col), d = E::ld(a.dy, db + col), t = E::ld(a.ddx, tb + col);
            const float u = __fmul_rn(d, g);
            const float ee = fmaf(-r2a, x, t);
            E::st(a.d_dy, row * a.ldd_dy + col, fmaf(g * r, ee, (r * x) * q));
            const float inner = fmaf(x, bd, fmaf(c, t, u * A));
            E::st(a.dx, row * a.lddx + col, fmaf(k5, x, fmaf(-r3, inner, (r * q) * d)));
            acc[col] = fmaf(r * d, ee, acc[col]);
        }
    }
    griddep_launch_dependents();
    if (blockIdx.x < a.M) {
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
        for (int col = tid; col < N; col += nt) wrow[col] = acc[col];
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool OFF, bool CL>
static const void* dbwd_tma_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&dbwd_tma_kernel<DT, 1, OFF, CL>);
    case 2: return reinterpret_cast<const void*>(&dbwd_tma_kernel<DT, 2, OFF, CL>);
    case 4: return reinterpret_cast<const void*>(&dbwd_tma_kernel<DT, 4, OFF, CL>);
    default: return nullptr;
    }
}
template <int DT, bool OFF>
static const void* dbwd_for(const Plan& p) {
    if (p.path == kPathScalar) return reinterpret_cast<const void*>(&dbwd_scalar_kernel<DT, OFF>);
    if (p.path == kPathRagged) return dbwd_ragged_kernel_ptr(p);
    if (p.path == kPathLanes) return lanes_kernel(4, p);
    if (p.path != kPathTma) return nullptr;
    return p.cluster > 1 ? dbwd_tma_vpt<DT, OFF, true>(p.per_thread) : dbwd_tma_vpt<DT, OFF, false>(p.per_thread);
}
template <bool OFF>
static const void* dbwd_pick(const Plan& p) {
    switch (p.dtype) {
    case kF32: return dbwd_for<kF32, OFF>(p);
    case kF16: return dbwd_for<kF16, OFF>(p);
    case kBF16: return dbwd_for<kBF16, OFF>(p);
    default: return nullptr;
    }
}

const void* dbwd_kernel(const Plan& p) { return p.offset ? dbwd_pick<true>(p) : dbwd_pick<false>(p); }

}  // namespace rmsnorm
