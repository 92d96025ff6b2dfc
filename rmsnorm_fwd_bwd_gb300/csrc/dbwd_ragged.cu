// dbwd_ragged.cu -- RMSNorm double backward (formulas of dbwd.cu) on the TMA ring
// for rows that do not start on a 16-byte boundary, with the row copies of
// ragged.cu: one ring stage holds the aligned spans of a row of x, dy and ddx
// (the three share their 16-byte phase), the neighbouring rows' elements of the
// first and last vector are masked to zero in registers, and (grid a multiple of
// 8) every row of a block starts at one phase, so each thread owns the same
// columns in all of them. g (or 1 + w) and ddgamma sit in shared memory as fp32
// float4 planes by vector slot (zero outside the row); the four row sums take one
// barrier; d_dy and d_x leave with 16-byte stores for whole vectors at their own
// row's phase and element stores otherwise; the d_gamma sums stay in registers.
#include "device.cuh"
#include "launch.h"
#include "ragged.cuh"

namespace rmsnorm {

// No register cap beyond the block size: capped at 96 registers (two blocks of
// 320 threads) bf16 N = 4099 ran at 4096 GB/s and fp32 at 4214, against 4785
// and 5539 with the compiler's own choice (159 and 132 registers).
template <int DT, int VPT, bool OFFSET>
__global__ void __launch_bounds__(kRaggedDbwdMaxThreads) dbwd_ragged_kernel(const RowArgs a) {
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
    const size_t t_pitch = static_cast<size_t>(a.ldddx) * E::kBytes;
    const size_t odx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const size_t ody_pitch = static_cast<size_t>(a.ldd_dy) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    const char* dyb = static_cast<const char*>(a.dy);
    const char* tb = static_cast<const char*>(a.ddx);
    char* odxb = static_cast<char*>(a.dx);
    char* odyb = static_cast<char*>(a.d_dy);
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * x_pitch) & 15);
    const int nv = static_cast<int>((static_cast<size_t>(o) + rowb + 15) / 16);
    const uint32_t span = static_cast<uint32_t>(nv) * 16;
    const uint32_t stride = (static_cast<uint32_t>(rowb) + 31) / 16 * 16;
    const int nslot = static_cast<int>(stride / 16);
    const int S = a.stages;

    // shared memory: ring (x, dy, ddx spans per stage) | g planes | ddgamma planes |
    // mbarriers | partials [2][4][32] | abort flag
    unsigned char* ring = smem;
    float4* gsm4 = reinterpret_cast<float4*>(smem + static_cast<size_t>(S) * 3 * stride);
    float4* qsm4 = gsm4 + (VEC / 4) * nslot;
    uint64_t* full = reinterpret_cast<uint64_t*>(qsm4 + (VEC / 4) * nslot);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 256);

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
        mbar_arrive_expect_tx(bar, 3 * span);
        bulk_g2s_in(smem_u32(st), xb + row * x_pitch - o, span, bar, pol, a.x, a.M, a.ldx, a.N, E::kBytes, a.err);
        bulk_g2s_in(smem_u32(st + stride), dyb + row * dy_pitch - o, span, bar, pol,
                    a.dy, a.M, a.lddy, a.N, E::kBytes, a.err);
        bulk_g2s_in(smem_u32(st + 2 * stride), tb + row * t_pitch - o, span, bar, pol,
                    a.ddx, a.M, a.ldddx, a.N, E::kBytes, a.err);
    };
    if (tid == 0) {
        const int64_t pre = nrows < S ? nrows : S;
        for (int64_t j = 0; j < pre; ++j) issue(j, ring + j * 3 * stride, smem_u32(&full[j]));
    }

    for (int idx = tid; idx < nslot; idx += nt) {
        int c0;
        const unsigned b = ragged::slot_bits<DT>(idx, nv, o, N, c0);
        float w[VEC], q[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = (b >> e) & 1u;
            const float g = in ? E::ld(a.gamma, c0 + e) : 0.f;
            w[e] = in ? (OFFSET ? 1.0f + g : g) : 0.f;
            q[e] = (in && a.ddg) ? E::ld(a.ddg, c0 + e) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < VEC; k += 4) {
            gsm4[(k / 4) * nslot + idx] = make_float4(w[k], w[k + 1], w[k + 2], w[k + 3]);
            qsm4[(k / 4) * nslot + idx] = make_float4(q[k], q[k + 1], q[k + 2], q[k + 3]);
        }
    }
    unsigned bits[VPT];
    float acc[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        int c0;
        bits[v] = ragged::slot_bits<DT>(v * nt + tid, nv, o, N, c0);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;
    }
    __syncthreads();

    auto rstd_at = [&](int64_t jj) -> float {
        return jj < nrows ? __ldg(a.rstd_in + blockIdx.x + jj * static_cast<int64_t>(gridDim.x)) : 0.f;
    };
    float r_cur = rstd_at(lane);
    float r_next = rstd_at(32 + lane);

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = blockIdx.x + j * static_cast<int64_t>(gridDim.x);
        const unsigned char* st = ring + static_cast<size_t>(s) * 3 * stride;
        if ((j & 31) == 0 && j > 0) {
            r_cur = r_next;
            r_next = rstd_at(j + 32 + lane);
        }
        const float r = __shfl_sync(0xffffffffu, r_cur, static_cast<int>(j & 31));
        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        // x, dy and ddx kept as their raw 16-byte words; the four row sums
        uint4 xs[VPT], ds[VPT], ts[VPT];
        float pc = 0.f, pa = 0.f, pb = 0.f, pd = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            xs[v] = ragged::slot_load<DT>(st, idx, bits[v]);
            ds[v] = ragged::slot_load<DT>(st + stride, idx, bits[v]);
            ts[v] = ragged::slot_load<DT>(st + 2 * stride, idx, bits[v]);
            if (bits[v] == 0u) continue;
            float xf[VEC], df[VEC], tf[VEC];
            E::unpack(xs[v], xf);
            E::unpack(ds[v], df);
            E::unpack(ts[v], tf);
#pragma unroll
            for (int k = 0; k < VEC; k += 4) {
                const float4 g4 = gsm4[(k / 4) * nslot + idx];
                const float4 q4 = qsm4[(k / 4) * nslot + idx];
                const float g[4] = {g4.x, g4.y, g4.z, g4.w};
                const float q[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = xf[k + e], d = df[k + e], t = tf[k + e];
                    const float u = __fmul_rn(d, g[e]);
                    pc = fmaf(u, x, pc);
                    pa = fmaf(t, x, pa);
                    pb = fmaf(t, u, pb);
                    pd = fmaf(__fmul_rn(q[e], d), x, pd);
                }
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
        __syncthreads();  // every thread has its words in registers: the stage can refill
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
        const float inv_n = 1.0f / static_cast<float>(N);
        const float c = warp_allsum(lane < nwarps ? redb[lane] : 0.f) * inv_n;
        const float A = warp_allsum(lane < nwarps ? redb[32 + lane] : 0.f) * inv_n;
        const float bd = (warp_allsum(lane < nwarps ? redb[64 + lane] : 0.f) +
                          warp_allsum(lane < nwarps ? redb[96 + lane] : 0.f)) * inv_n;  // B + D
        const float r2 = r * r;
        const float r3 = r2 * r;
        const float r2a = r2 * A;
        const float k5 = (3.0f * (r3 * r2)) * (c * A);

        if (!aborted) {
            char* odx_row = odxb + static_cast<size_t>(row) * odx_pitch;
            char* ody_row = odyb + static_cast<size_t>(row) * ody_pitch;
            const bool x_phase = (reinterpret_cast<uintptr_t>(odx_row) & 15) == static_cast<uintptr_t>(o);
            const bool y_phase = (reinterpret_cast<uintptr_t>(ody_row) & 15) == static_cast<uintptr_t>(o);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (bits[v] == 0u) continue;
                const int idx = v * nt + tid;
                float xf[VEC], df[VEC], tf[VEC], o_dy[VEC], o_x[VEC];
                E::unpack(xs[v], xf);
                E::unpack(ds[v], df);
                E::unpack(ts[v], tf);
#pragma unroll
                for (int k = 0; k < VEC; k += 4) {
                    const float4 g4 = gsm4[(k / 4) * nslot + idx];
                    const float4 q4 = qsm4[(k / 4) * nslot + idx];
                    const float g[4] = {g4.x, g4.y, g4.z, g4.w};
                    const float q[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x = xf[k + e], d = df[k + e], t = tf[k + e];
                        const float u = __fmul_rn(d, g[e]);
                        const float ee = fmaf(-r2a, x, t);  // ddx - r^2 x A
                        o_dy[k + e] = fmaf(g[e] * r, ee, (r * x) * q[e]);
                        const float inner = fmaf(x, bd, fmaf(c, t, u * A));
                        o_x[k + e] = fmaf(k5, x, fmaf(-r3, inner, (r * q[e]) * d));
                        acc[v][k + e] = fmaf(r * d, ee, acc[v][k + e]);
                    }
                }
                const int c0 = (16 * idx - o) / E::kBytes;
                if (bits[v] == kAll && y_phase) {
                    stg128(ody_row - o + idx * 16, E::pack(o_dy));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if ((bits[v] >> e) & 1u) E::st(ody_row, c0 + e, o_dy[e]);
                }
                if (bits[v] == kAll && x_phase) {
                    stg128(odx_row - o + idx * 16, E::pack(o_x));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if ((bits[v] >> e) & 1u) E::st(odx_row, c0 + e, o_x[e]);
                }
            }
        }
    }
    griddep_launch_dependents();
    // one row of d_gamma partials per block (zeros for a block without rows)
    if (!aborted) {
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c0 = (16 * (v * nt + tid) - o) / E::kBytes;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if ((bits[v] >> e) & 1u) wrow[c0 + e] = acc[v][e];
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
// Instances up to 24 elements per thread (the planner's register budget for
// this kernel): 2-byte types up to 3 vectors, fp32 up to 6.
template <int DT, int VPT, bool OFF>
static const void* dbwd_ragged_entry() {
    if constexpr (VPT * Elem<DT>::kVec <= 24) return reinterpret_cast<const void*>(&dbwd_ragged_kernel<DT, VPT, OFF>);
    else return nullptr;
}
template <int DT, bool OFF>
static const void* dbwd_ragged_pick(int vpt) {
    switch (vpt) {
    case 1: return dbwd_ragged_entry<DT, 1, OFF>();
    case 2: return dbwd_ragged_entry<DT, 2, OFF>();
    case 3: return dbwd_ragged_entry<DT, 3, OFF>();
    case 4: return dbwd_ragged_entry<DT, 4, OFF>();
    case 5: return dbwd_ragged_entry<DT, 5, OFF>();
    case 6: return dbwd_ragged_entry<DT, 6, OFF>();
    default: return nullptr;
    }
}

const void* dbwd_ragged_kernel_ptr(const Plan& p) {
    switch (p.dtype) {
    case kF32: return p.offset ? dbwd_ragged_pick<kF32, true>(p.per_thread) : dbwd_ragged_pick<kF32, false>(p.per_thread);
    case kF16: return p.offset ? dbwd_ragged_pick<kF16, true>(p.per_thread) : dbwd_ragged_pick<kF16, false>(p.per_thread);
    case kBF16:
        return p.offset ? dbwd_ragged_pick<kBF16, true>(p.per_thread) : dbwd_ragged_pick<kBF16, false>(p.per_thread);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
