// ln_bwd.cu -- LayerNorm backward kernels.
//
// Per row, with mu and r saved by the forward, x_hat = (x - mu) * r and
// u = dy * gamma (the standard LayerNorm gradient; page "torch.compile
// performance leap: optimizing LayerNorm and RMSNorm kernels", section 2 names
// the three gradients -- input, weight and bias -- and section 2.1 the fused
// kernel that reduces rows for dx and columns for dgamma and dbeta while
// reading the inputs once):
//     dx = r * ((u - mean_j u_j) - x_hat * mean_j(u_j * x_hat_j))
//     dgamma_j = sum over rows of dy_j * x_hat_j;   dbeta_j = sum over rows of dy_j
//
// Same structure as the RMSNorm backward: one fused row kernel (x and dy read
// once through the TMA ring, dx written, two row sums reduced with one barrier,
// per-block fp32 column accumulators for dgamma and dbeta in registers) that
// leaves one row of dgamma partials and one row of dbeta partials per block in
// the workspace, then the fixed-order column reduce for both (deterministic,
// no floating-point atomics). Workspace: 2 x units x N floats.
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

template <int DT, int VPT, bool CLUSTER>
__global__ void __launch_bounds__(kTmaMaxThreads) ln_bwd_tma_kernel(const RowArgs a) {
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

    // shared memory: ring | gamma slice in fp32 | mbarriers | warp partials [2][2][32] | abort flag
    unsigned char* ring = smem;
    float* gsm = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(gsm + ns);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 128);

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

    // gamma slice widened once into shared memory as VEC/4 planes of float4
    float4* gsm4 = reinterpret_cast<float4*>(gsm);
    {
        const uint4* gs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.gamma) + slice_off);
        for (int idx = tid; idx < nvec; idx += nt) {
            float w[VEC];
            E::unpack(__ldg(gs + idx), w);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) gsm4[(q / 4) * nvec + idx] = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
        }
    }
    float accg[VPT][VEC], accb[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int e = 0; e < VEC; ++e) accg[v][e] = accb[v][e] = 0.f;

    __syncthreads();
    if (CLUSTER) cluster_sync();

    // saved mean and r, 32 rows per warp-wide load, fetched 32 rows ahead of use
    auto saved_at = [&](const float* p, int64_t jj) -> float {
        return jj < nrows ? __ldg(p + cid + jj * ncl) : 0.f;
    };
    float m_cur = saved_at(a.mean_in, lane), m_next = saved_at(a.mean_in, 32 + lane);
    float r_cur = saved_at(a.rstd_in, lane), r_next = saved_at(a.rstd_in, 32 + lane);

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = cid + j * ncl;
        const unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
        if ((j & 31) == 0 && j > 0) {
            m_cur = m_next;
            r_cur = r_next;
            m_next = saved_at(a.mean_in, j + 32 + lane);
            r_next = saved_at(a.rstd_in, j + 32 + lane);
        }
        const float mu = __shfl_sync(0xffffffffu, m_cur, static_cast<int>(j & 31));
        const float r = __shfl_sync(0xffffffffu, r_cur, static_cast<int>(j & 31));

        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        // x_hat and u kept in registers; sums of u and u * x_hat; column terms
        float hf[VPT][VEC], uf[VPT][VEC];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            float xf[VEC], df[VEC], g[VEC];
            if (idx < nvec) {
                E::unpack(*reinterpret_cast<const uint4*>(st + idx * 16), xf);
                E::unpack(*reinterpret_cast<const uint4*>(st + slice_bytes + idx * 16), df);
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    const float4 f = gsm4[(q / 4) * nvec + idx];
                    g[q] = f.x; g[q + 1] = f.y; g[q + 2] = f.z; g[q + 3] = f.w;
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    hf[v][e] = __fmul_rn(xf[e] - mu, r);
                    uf[v][e] = __fmul_rn(df[e], g[e]);
                    p0 += uf[v][e];
                    p1 = fmaf(uf[v][e], hf[v][e], p1);
                    accg[v][e] = fmaf(df[e], hf[v][e], accg[v][e]);
                    accb[v][e] += df[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) hf[v][e] = uf[v][e] = 0.f;
            }
        }
        float* redb = red + (j & 1) * 64;
        const float w0 = warp_allsum(p0);
        const float w1 = warp_allsum(p1);
        if (lane == 0) {
            redb[warp] = w0;
            redb[32 + warp] = w1;
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

        float t0 = 0.f, t1 = 0.f;
        if (!CLUSTER) {
            if (lane < nwarps) {
                t0 = redb[lane];
                t1 = redb[32 + lane];
            }
        } else if (lane < nwarps * static_cast<int>(csize)) {
            const uint32_t rk = static_cast<uint32_t>(lane / nwarps);
            const int w = lane % nwarps;
            t0 = dsmem_ld_f32(dsmem_map(smem_u32(redb + w), rk));
            t1 = dsmem_ld_f32(dsmem_map(smem_u32(redb + 32 + w), rk));
        }
        const float c1 = warp_allsum(t0) / static_cast<float>(a.N);  // mean(u)
        const float c2 = warp_allsum(t1) / static_cast<float>(a.N);  // mean(u * x_hat)

        if (!aborted) {
            char* dxrow = dxsl + static_cast<size_t>(row) * dx_pitch;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int idx = v * nt + tid;
                if (idx < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = r * fmaf(-hf[v][e], c2, uf[v][e] - c1);
                    stg128(dxrow + idx * 16, E::pack(o));
                }
            }
        }
    }

    griddep_launch_dependents();
    // one row of dgamma partials (plane 0) and of dbeta partials (plane 1) per cluster
    if (!aborted) {
        const size_t plane = static_cast<size_t>(ncl) * a.ldws;
        float* wrow = a.ws + static_cast<size_t>(cid) * a.ldws + static_cast<size_t>(crank) * ns;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            if (idx < nvec) {
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    *reinterpret_cast<float4*>(wrow + idx * VEC + q) =
                        make_float4(accg[v][q], accg[v][q + 1], accg[v][q + 2], accg[v][q + 3]);
                    *reinterpret_cast<float4*>(wrow + plane + idx * VEC + q) =
                        make_float4(accb[v][q], accb[v][q + 1], accb[v][q + 2], accb[v][q + 3]);
                }
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

// General path: any N, any element alignment. One CTA per row (persistent);
// thread t owns columns t, t + nt, ...; two passes over the row (the second is
// served by L1/L2); dgamma and dbeta accumulators live in shared memory
// indexed by column (each column is touched by one thread only).
template <int DT>
__global__ void __launch_bounds__(kScalarThreads) ln_bwd_scalar_kernel(const RowArgs a) {
    using E = Elem<DT>;
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N;
    float* accg = reinterpret_cast<float*>(smem);  // [N]
    float* accb = accg + N;                        // [N]
    __shared__ float red[2][2][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    griddep_wait();

    for (int c = tid; c < N; c += nt) accg[c] = accb[c] = 0.f;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t base = row * a.ldx;
        const int64_t dbase = row * a.lddy;
        const int64_t obase = row * a.lddx;
        const float mu = __ldg(a.mean_in + row);
        const float r = __ldg(a.rstd_in + row);
        float p0 = 0.f, p1 = 0.f;
        for (int col = tid; col < N; col += nt) {
            const float xh = __fmul_rn(E::ld(a.x, base + col) - mu, r);
            const float d = E::ld(a.dy, dbase + col);
            const float u = __fmul_rn(d, E::ld(a.gamma, col));
            p0 += u;
            p1 = fmaf(u, xh, p1);
            accg[col] = fmaf(d, xh, accg[col]);
            accb[col] += d;
        }
        const float w0 = warp_allsum(p0);
        const float w1 = warp_allsum(p1);
        if (lane == 0) {
            red[parity][0][warp] = w0;
            red[parity][1][warp] = w1;
        }
        __syncthreads();
        const float t0 = lane < nwarps ? red[parity][0][lane] : 0.f;
        const float t1 = lane < nwarps ? red[parity][1][lane] : 0.f;
        const float c1 = warp_allsum(t0) / static_cast<float>(N);
        const float c2 = warp_allsum(t1) / static_cast<float>(N);
#pragma unroll 4
        for (int c = tid; c < N; c += nt) {
            const float xh = __fmul_rn(E::ld(a.x, base + c) - mu, r);
            const float u = __fmul_rn(E::ld(a.dy, dbase + c), E::ld(a.gamma, c));
            E::st(a.dx, obase + c, r * fmaf(-xh, c2, u - c1));
        }
    }
    griddep_launch_dependents();
    if (blockIdx.x < a.M) {
        const size_t plane = static_cast<size_t>(gridDim.x) * a.ldws;
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
        for (int c = tid; c < N; c += nt) {
            wrow[c] = accg[c];
            wrow[plane + c] = accb[c];
        }
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool CL>
static const void* ln_bwd_tma_vpt(int vpt) {
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&ln_bwd_tma_kernel<DT, 1, CL>);
    case 2: return reinterpret_cast<const void*>(&ln_bwd_tma_kernel<DT, 2, CL>);
    case 4: return reinterpret_cast<const void*>(&ln_bwd_tma_kernel<DT, 4, CL>);
    case 8: return reinterpret_cast<const void*>(&ln_bwd_tma_kernel<DT, 8, CL>);
    default: return nullptr;
    }
}
template <int DT>
static const void* ln_bwd_for(const Plan& p) {
    if (p.path == kPathScalar) return reinterpret_cast<const void*>(&ln_bwd_scalar_kernel<DT>);
    if (p.path != kPathTma) return nullptr;
    return p.cluster > 1 ? ln_bwd_tma_vpt<DT, true>(p.per_thread) : ln_bwd_tma_vpt<DT, false>(p.per_thread);
}

const void* ln_bwd_kernel(const Plan& p) {
    if (p.path == kPathLanes) return lanes_kernel(3, p);
    if (p.path == kPathRowVec) return ln_rowvec_kernel(3, p);
    if (p.path == kPathRagged) return ln_ragged_kernel(3, p);
    switch (p.dtype) {
    case kF32: return ln_bwd_for<kF32>(p);
    case kF16: return ln_bwd_for<kF16>(p);
    case kBF16: return ln_bwd_for<kBF16>(p);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
