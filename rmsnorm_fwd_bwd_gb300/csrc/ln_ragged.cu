// ln_ragged.cu -- LayerNorm forward and backward on the TMA ring for rows that do
// not start on a 16-byte boundary, with the formulas of ln_fwd.cu and ln_bwd.cu
// and the row copies of ragged.cu: one bulk copy of each row's aligned span
// into a shared-memory ring, the neighbouring rows' elements of the first and
// last vector masked to zero in registers, and (grid a multiple of 8) one
// 16-byte phase per block, so every thread owns the same columns in all rows of
// its block. gamma and beta sit in shared memory as fp32 float4 planes by vector
// slot; the forward counts each warp's elements once and takes its statistics
// with one barrier per row (warp two-pass, then the parallel-axis combination);
// the backward keeps its dgamma and dbeta sums in registers.
#include "device.cuh"
#include "launch.h"
#include "ragged.cuh"

namespace rmsnorm {

namespace {

// fp32 planes of a per-column vector by slot, zero outside the row
template <int DT>
__device__ __forceinline__ void stage_slots(const void* src, int N, int o, int nv, int nslot, float4* dst) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    for (int idx = threadIdx.x; idx < nslot; idx += blockDim.x) {
        int c0;
        const unsigned b = ragged::slot_bits<DT>(idx, nv, o, N, c0);
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = ((b >> e) & 1u) ? E::ld(src, c0 + e) : 0.f;
#pragma unroll
        for (int q = 0; q < VEC; q += 4) dst[(q / 4) * nslot + idx] = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
    }
}

}  // namespace

template <int DT, int VPT>
__global__ void __launch_bounds__(kTmaMaxThreads, 3) ln_fwd_ragged_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr unsigned kAll = (1u << VEC) - 1u;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    const size_t rowb = static_cast<size_t>(N) * E::kBytes;
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    char* yb = static_cast<char*>(a.y);
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * x_pitch) & 15);
    const int nv = static_cast<int>((static_cast<size_t>(o) + rowb + 15) / 16);
    const uint32_t span = static_cast<uint32_t>(nv) * 16;
    const uint32_t stride = (static_cast<uint32_t>(rowb) + 31) / 16 * 16;
    const int nslot = static_cast<int>(stride / 16);
    const int S = a.stages;

    // shared memory: ring | gamma planes | beta planes | mbarriers | partials n, m, q [2][32] | abort
    unsigned char* ring = smem;
    float4* gsm4 = reinterpret_cast<float4*>(smem + static_cast<size_t>(S) * stride);
    float4* bsm4 = gsm4 + (VEC / 4) * nslot;
    uint64_t* full = reinterpret_cast<uint64_t*>(bsm4 + (VEC / 4) * nslot);
    float* red_n = reinterpret_cast<float*>(full + S);
    float* red_m = red_n + 64;
    float* red_q = red_n + 128;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red_n + 192);

    const int64_t nrows = blockIdx.x < a.M ? (a.M - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_wait();
    // the first rows' copies go out before the per-column set-up below, so the
    // ring fills while gamma is being loaded
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t j, const unsigned char* st, uint32_t bar) {
        const size_t row = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(j) * gridDim.x;
        mbar_arrive_expect_tx(bar, span);
        bulk_g2s_in(smem_u32(st), xb + row * x_pitch - o, span, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
    };
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) issue(j, ring + j * stride, smem_u32(&full[j]));
    }
    stage_slots<DT>(a.gamma, N, o, nv, nslot, gsm4);
    stage_slots<DT>(a.beta, N, o, nv, nslot, bsm4);
    unsigned bits[VPT];
    int cnt = 0;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        int c0;
        bits[v] = ragged::slot_bits<DT>(v * nt + tid, nv, o, N, c0);
        cnt += __popc(bits[v]);
    }
    const float n_warp = warp_allsum(static_cast<float>(cnt));
    __syncthreads();

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = blockIdx.x + j * static_cast<int64_t>(gridDim.x);
        const unsigned char* st = ring + static_cast<size_t>(s) * stride;
        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        // the warp's mean (masked elements are zero), then its squared deviations
        float xf[VPT][VEC];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            E::unpack(ragged::slot_load<DT>(st, v * nt + tid, bits[v]), xf[v]);
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
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float d = ((bits[v] >> e) & 1u) ? xf[v][e] - m_warp : 0.f;
                if (e & 1) q1 = fmaf(d, d, q1); else q0 = fmaf(d, d, q0);
            }
        }
        const float q_warp = warp_allsum(q0 + q1);
        const int b = static_cast<int>(j & 1) * 32;
        if (lane == 0) {
            red_n[b + warp] = n_warp;
            red_m[b + warp] = m_warp;
            red_q[b + warp] = q_warp;
        }
        __syncthreads();  // every thread has its slots in registers: the stage can refill
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
        const float tn = lane < nwarps ? red_n[b + lane] : 0.f;
        const float tm = lane < nwarps ? red_m[b + lane] : 0.f;
        const float tq = lane < nwarps ? red_q[b + lane] : 0.f;
        const float mu = warp_allsum(tn * tm) / static_cast<float>(N);
        const float dm = tm - mu;
        const float var = warp_allsum(fmaf(tn * dm, dm, tq)) / static_cast<float>(N);
        const float r = 1.0f / sqrtf(var + a.eps);

        if (!aborted) {
            if (tid == 0) {
                if (a.mean_out) a.mean_out[row] = mu;
                if (a.rstd_out) a.rstd_out[row] = r;
            }
            char* yrow = yb + static_cast<size_t>(row) * y_pitch;
            const bool same_phase = (reinterpret_cast<uintptr_t>(yrow) & 15) == static_cast<uintptr_t>(o);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (bits[v] == 0u) continue;
                const int idx = v * nt + tid;
                float out[VEC];
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    const float4 g4 = gsm4[(q / 4) * nslot + idx];
                    const float4 b4 = bsm4[(q / 4) * nslot + idx];
                    out[q] = fmaf((xf[v][q] - mu) * r, g4.x, b4.x);
                    out[q + 1] = fmaf((xf[v][q + 1] - mu) * r, g4.y, b4.y);
                    out[q + 2] = fmaf((xf[v][q + 2] - mu) * r, g4.z, b4.z);
                    out[q + 3] = fmaf((xf[v][q + 3] - mu) * r, g4.w, b4.w);
                }
                if (bits[v] == kAll && same_phase) {
                    stg128(yrow - o + idx * 16, E::pack(out));
                } else {
                    const int c0 = (16 * idx - o) / E::kBytes;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if ((bits[v] >> e) & 1u) E::st(yrow, c0 + e, out[e]);
                }
            }
        }
    }
    griddep_launch_dependents();
    if (aborted && tid == 0) {
        const int64_t end = abort_row + S < nrows ? abort_row + S : nrows;
        for (int64_t j = abort_row; j < end; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), static_cast<uint32_t>((j / S) & 1), a.err, 1u << 16);
    }
}

template <int DT, int VPT>
__global__ void __launch_bounds__(kTmaMaxThreads) ln_bwd_ragged_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr unsigned kAll = (1u << VEC) - 1u;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    const size_t rowb = static_cast<size_t>(N) * E::kBytes;
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
    const size_t dx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    const char* dyb = static_cast<const char*>(a.dy);
    char* dxb = static_cast<char*>(a.dx);
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * x_pitch) & 15);
    const int nv = static_cast<int>((static_cast<size_t>(o) + rowb + 15) / 16);
    const uint32_t span = static_cast<uint32_t>(nv) * 16;
    const uint32_t stride = (static_cast<uint32_t>(rowb) + 31) / 16 * 16;
    const int nslot = static_cast<int>(stride / 16);
    const int S = a.stages;

    // shared memory: ring (x span, dy span per stage) | gamma planes | mbarriers | partials [2][2][32] | abort
    unsigned char* ring = smem;
    float4* gsm4 = reinterpret_cast<float4*>(smem + static_cast<size_t>(S) * 2 * stride);
    uint64_t* full = reinterpret_cast<uint64_t*>(gsm4 + (VEC / 4) * nslot);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 128);

    const int64_t nrows = blockIdx.x < a.M ? (a.M - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_wait();
    // the first rows' copies go out before the per-column set-up below, so the
    // ring fills while gamma is being loaded
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t j, const unsigned char* st, uint32_t bar) {
        const size_t row = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(j) * gridDim.x;
        mbar_arrive_expect_tx(bar, 2 * span);
        bulk_g2s_in(smem_u32(st), xb + row * x_pitch - o, span, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
        bulk_g2s_in(smem_u32(st + stride), dyb + row * dy_pitch - o, span, bar, pol,
                    a.dy, a.M, a.lddy, a.N, E::kBytes, a.err);
    };
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) issue(j, ring + j * 2 * stride, smem_u32(&full[j]));
    }
    stage_slots<DT>(a.gamma, N, o, nv, nslot, gsm4);
    unsigned bits[VPT];
    float accg[VPT][VEC], accb[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        int c0;
        bits[v] = ragged::slot_bits<DT>(v * nt + tid, nv, o, N, c0);
#pragma unroll
        for (int e = 0; e < VEC; ++e) accg[v][e] = accb[v][e] = 0.f;
    }
    __syncthreads();

    auto saved_at = [&](const float* p, int64_t jj) -> float {
        return jj < nrows ? __ldg(p + blockIdx.x + jj * static_cast<int64_t>(gridDim.x)) : 0.f;
    };
    float m_cur = saved_at(a.mean_in, lane), m_next = saved_at(a.mean_in, 32 + lane);
    float r_cur = saved_at(a.rstd_in, lane), r_next = saved_at(a.rstd_in, 32 + lane);

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = blockIdx.x + j * static_cast<int64_t>(gridDim.x);
        const unsigned char* st = ring + static_cast<size_t>(s) * 2 * stride;
        if ((j & 31) == 0 && j > 0) {
            m_cur = m_next;
            r_cur = r_next;
            m_next = saved_at(a.mean_in, j + 32 + lane);
            r_next = saved_at(a.rstd_in, j + 32 + lane);
        }
        const float mu = __shfl_sync(0xffffffffu, m_cur, static_cast<int>(j & 31));
        const float r = __shfl_sync(0xffffffffu, r_cur, static_cast<int>(j & 31));
        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        // x_hat and u = dy * gamma; outside the row x, dy and gamma are zero, so u and
        // every product with dy vanish there whatever x_hat is (-mean * r), and
        // those columns are never written: x_hat needs no mask
        float hf[VPT][VEC], uf[VPT][VEC];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            float xf[VEC], df[VEC], g[VEC];
            E::unpack(ragged::slot_load<DT>(st, idx, bits[v]), xf);
            E::unpack(ragged::slot_load<DT>(st + stride, idx, bits[v]), df);
            if (bits[v]) {
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                    const float4 f = gsm4[(q / 4) * nslot + idx];
                    g[q] = f.x; g[q + 1] = f.y; g[q + 2] = f.z; g[q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) g[e] = 0.f;
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
        }
        float* redb = red + (j & 1) * 64;
        const float w0 = warp_allsum(p0);
        const float w1 = warp_allsum(p1);
        if (lane == 0) {
            redb[warp] = w0;
            redb[32 + warp] = w1;
        }
        __syncthreads();
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
        const float c1 = warp_allsum(lane < nwarps ? redb[lane] : 0.f) / static_cast<float>(N);
        const float c2 = warp_allsum(lane < nwarps ? redb[32 + lane] : 0.f) / static_cast<float>(N);

        if (!aborted) {
            char* dxrow = dxb + static_cast<size_t>(row) * dx_pitch;
            const bool same_phase = (reinterpret_cast<uintptr_t>(dxrow) & 15) == static_cast<uintptr_t>(o);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (bits[v] == 0u) continue;
                const int idx = v * nt + tid;
                float out[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) out[e] = r * fmaf(-hf[v][e], c2, uf[v][e] - c1);
                if (bits[v] == kAll && same_phase) {
                    stg128(dxrow - o + idx * 16, E::pack(out));
                } else {
                    const int c0 = (16 * idx - o) / E::kBytes;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if ((bits[v] >> e) & 1u) E::st(dxrow, c0 + e, out[e]);
                }
            }
        }
    }
    griddep_launch_dependents();
    // one row of dgamma partials (plane 0) and dbeta partials (plane 1) per block
    if (!aborted) {
        const size_t plane = static_cast<size_t>(gridDim.x) * a.ldws;
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c0 = (16 * (v * nt + tid) - o) / E::kBytes;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if ((bits[v] >> e) & 1u) {
                    wrow[c0 + e] = accg[v][e];
                    wrow[plane + c0 + e] = accb[v][e];
                }
        }
    }
    if (aborted && tid == 0) {
        const int64_t end = abort_row + S < nrows ? abort_row + S : nrows;
        for (int64_t j = abort_row; j < end; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), static_cast<uint32_t>((j / S) & 1), a.err, 1u << 16);
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT>
static const void* ln_ragged_pick(int pass, int vpt) {
#define LAYERNORM_RG(V)                                                                  \
    case V:                                                                              \
        return pass == 2 ? reinterpret_cast<const void*>(&ln_fwd_ragged_kernel<DT, V>)   \
                         : reinterpret_cast<const void*>(&ln_bwd_ragged_kernel<DT, V>);
    switch (vpt) {
        LAYERNORM_RG(1)
        LAYERNORM_RG(2)
        LAYERNORM_RG(3)
        LAYERNORM_RG(4)
        LAYERNORM_RG(5)
        LAYERNORM_RG(6)
    default: return nullptr;
    }
#undef LAYERNORM_RG
}

const void* ln_ragged_kernel(int pass, const Plan& p) {
    if (pass != 2 && pass != 3) return nullptr;
    switch (p.dtype) {
    case kF32: return ln_ragged_pick<kF32>(pass, p.per_thread);
    case kF16: return ln_ragged_pick<kF16>(pass, p.per_thread);
    case kBF16: return ln_ragged_pick<kBF16>(pass, p.per_thread);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
