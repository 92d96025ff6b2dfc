// ragged.cu -- RMSNorm forward and backward on the TMA ring for rows that do not
// start on a 16-byte boundary (N * sizeof(dtype) not a multiple of 16, e.g. bf16
// N = 4099, or pointers and pitches off 16 bytes), with the formulas of fwd.cu
// and bwd.cu.
//
// The grid is a multiple of 8, so every row of a persistent block (blockIdx.x
// + k * gridDim.x) starts at the same 16-byte phase o (rows r and r + 8 always
// share it). Each row is copied by one TMA bulk copy of its aligned span
// [row start - o, ceil16(row end)) -- nv 16-byte vectors, the same count for
// every row of the block -- into a shared-memory ring. Every 16-byte chunk of
// that span holds at least one byte of the tensor, so the copy never leaves the
// tensor's own chunks; the elements of neighbouring rows it brings along sit
// only in the first and last vector and are masked to zero in registers.
// Thread t owns vector slots t, t + nt, ... and so the same columns in every
// row of its block: gamma (forward: registers; backward: fp32 float4 planes in
// shared memory) and the backward's dgamma sums (registers) follow the slots.
// Outputs with the rows' phase get 16-byte stores for whole vectors and element
// stores at the two ends (a neighbour's elements are never written); outputs at
// another phase are written element by element. Waits are bounded as in the
// aligned TMA kernels.
#include "device.cuh"
#include "launch.h"
#include "ragged.cuh"

namespace rmsnorm {

// Minimum resident blocks passed to the forward's __launch_bounds__ (0: none):
// these instances fit 68 registers without spills when asked for three
// 256-thread blocks (e.g. three 192-thread blocks per SM for bf16 N = 4099);
// left alone ptxas uses 108 (two blocks).
template <int DT, int VPT> struct RaggedFwdMinBlocks { static constexpr int value = (VPT <= 3 || DT == kF32) ? 3 : 0; };

template <int DT, int VPT, bool OFFSET>
__global__ void __launch_bounds__(kTmaMaxThreads, (RaggedFwdMinBlocks<DT, VPT>::value))
    fwd_ragged_kernel(const RowArgs a) {
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
    const int nv = static_cast<int>((static_cast<size_t>(o) + rowb + 15) / 16);  // vectors of a row's span
    const uint32_t span = static_cast<uint32_t>(nv) * 16;
    const uint32_t stride = (static_cast<uint32_t>(rowb) + 31) / 16 * 16;  // ring stage size (any phase)
    const int S = a.stages;

    // shared memory: ring | mbarriers | warp partials [2][32] | abort flag
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stride);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

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

    // this thread's slots: which elements lie in the row, and gamma (or 1 + w) there
    unsigned bits[VPT];
    float gf[VPT][VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        int c0;
        bits[v] = ragged::slot_bits<DT>(v * nt + tid, nv, o, N, c0);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = (bits[v] >> e) & 1u;
            const float w = in ? E::ld(a.gamma, c0 + e) : 0.f;
            gf[v][e] = in ? (OFFSET ? 1.0f + w : w) : 0.f;
        }
    }
    __syncthreads();

    bool aborted = false;
    int64_t abort_row = nrows;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t j = 0; j < nrows; ++j) {
        const int64_t row = blockIdx.x + j * static_cast<int64_t>(gridDim.x);
        const unsigned char* st = ring + static_cast<size_t>(s) * stride;
        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        float xf[VPT][VEC];
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            E::unpack(ragged::slot_load<DT>(st, v * nt + tid, bits[v]), xf[v]);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                ss0 = fmaf(xf[v][e], xf[v][e], ss0);
                ss1 = fmaf(xf[v][e + 1], xf[v][e + 1], ss1);
            }
        }
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(ss0 + ss1);
        if (lane == 0) redb[warp] = wsum;
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
        float t = lane < nwarps ? redb[lane] : 0.f;
        t = warp_allsum(t);
        const float r = 1.0f / sqrtf(t / static_cast<float>(N) + a.eps);

        if (!aborted) {
            if (tid == 0) a.rstd_out[row] = r;
            char* yrow = yb + static_cast<size_t>(row) * y_pitch;
            const bool same_phase = (reinterpret_cast<uintptr_t>(yrow) & 15) == static_cast<uintptr_t>(o);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (bits[v] == 0u) continue;
                const int idx = v * nt + tid;
                // scalar form: the packed one (f32x2) measured slower here (bf16
                // 8192x4099 forward 29.2 -> 32.6 us), unlike the ring forward
                float out[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    out[e] = OFFSET ? (gf[v][e] * xf[v][e]) * r : (xf[v][e] * r) * gf[v][e];
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

template <int DT, int VPT, bool OFFSET>
__global__ void __launch_bounds__(kTmaMaxThreads) bwd_ragged_kernel(const RowArgs a) {
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
    // x and dy rows share their phase (same pointer phase, pitches equal modulo 16)
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * x_pitch) & 15);
    const int nv = static_cast<int>((static_cast<size_t>(o) + rowb + 15) / 16);
    const uint32_t span = static_cast<uint32_t>(nv) * 16;
    const uint32_t stride = (static_cast<uint32_t>(rowb) + 31) / 16 * 16;
    const int nslot = static_cast<int>(stride / 16);  // vector slots of any phase
    const int S = a.stages;

    // shared memory: ring (x span, dy span per stage) | gamma planes | mbarriers | partials [2][32] | abort
    unsigned char* ring = smem;
    float4* gsm4 = reinterpret_cast<float4*>(smem + static_cast<size_t>(S) * 2 * stride);
    uint64_t* full = reinterpret_cast<uint64_t*>(gsm4 + (VEC / 4) * nslot);
    float* red = reinterpret_cast<float*>(full + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);

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

    // gamma (or 1 + w) by vector slot at this block's phase, zero outside the row
    for (int idx = tid; idx < nslot; idx += nt) {
        int c0;
        const unsigned b = ragged::slot_bits<DT>(idx, nv, o, N, c0);
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = (b >> e) & 1u;
            const float g = in ? E::ld(a.gamma, c0 + e) : 0.f;
            w[e] = in ? (OFFSET ? 1.0f + g : g) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < VEC; q += 4) gsm4[(q / 4) * nslot + idx] = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
    }
    // 2-byte types with up to three vectors per thread run the arithmetic on
    // packed pairs (f32x2: one instruction for two elements, each rounded as the
    // scalar operation, so the same bits; bf16 8192x4099: 53.8 -> 52.4 us). With
    // more vectors the packed form needs more registers than the scalar one (bf16
    // 128 -> 132, fp16 128 -> 200) and would halve the blocks per SM, and for
    // fp32 ptxas spilled; those instances keep the scalar form.
    constexpr bool PACKED = VPT <= 3 && DT != kF32;
    unsigned bits[VPT];
    float acc[VPT][VEC];
    uint64_t acc2[PACKED ? VPT : 1][VEC / 2];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        int c0;
        bits[v] = ragged::slot_bits<DT>(v * nt + tid, nv, o, N, c0);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) acc2[PACKED ? v : 0][e] = f2_pack(0.f, 0.f);
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
        const unsigned char* st = ring + static_cast<size_t>(s) * 2 * stride;
        if ((j & 31) == 0 && j > 0) {
            r_cur = r_next;
            r_next = rstd_at(j + 32 + lane);
        }
        const float r = __shfl_sync(0xffffffffu, r_cur, static_cast<int>(j & 31));
        if (!aborted && !mbar_wait_bounded(smem_u32(&full[s]), parity, a.err)) *abort_flag = 1;

        float xf[PACKED ? 1 : VPT][VEC], uf[PACKED ? 1 : VPT][VEC];
        uint64_t x2[PACKED ? VPT : 1][VEC / 2], u2[PACKED ? VPT : 1][VEC / 2];
        float p0 = 0.f, p1 = 0.f;
        uint64_t p2 = f2_pack(0.f, 0.f);
        const uint64_t r2 = f2_pack(r, r);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            float xv[VEC], df[VEC];
            E::unpack(ragged::slot_load<DT>(st, idx, bits[v]), xv);
            E::unpack(ragged::slot_load<DT>(st + stride, idx, bits[v]), df);
            float g[VEC];
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
            if constexpr (PACKED) {
                // u = dy * g, the row sum of u * x in two lanes (even and odd elements)
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    const uint64_t xx = f2_pack(xv[e], xv[e + 1]);
                    const uint64_t dd = f2_pack(df[e], df[e + 1]);
                    const uint64_t uu = f2_mul(dd, f2_pack(g[e], g[e + 1]));
                    p2 = f2_fma(uu, xx, p2);
                    acc2[v][e / 2] = f2_fma(f2_mul(dd, xx), r2, acc2[v][e / 2]);
                    x2[v][e / 2] = xx;
                    u2[v][e / 2] = uu;
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    xf[v][e] = xv[e];
                    uf[v][e] = __fmul_rn(df[e], g[e]);
                    if (e & 1) p1 = fmaf(uf[v][e], xv[e], p1); else p0 = fmaf(uf[v][e], xv[e], p0);
                    acc[v][e] = fmaf(__fmul_rn(df[e], xv[e]), r, acc[v][e]);
                }
            }
        }
        if constexpr (PACKED) f2_unpack(p2, p0, p1);
        float* redb = red + (j & 1) * 32;
        const float wsum = warp_allsum(p0 + p1);
        if (lane == 0) redb[warp] = wsum;
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
        float t = lane < nwarps ? redb[lane] : 0.f;
        t = warp_allsum(t);
        const float c = t / static_cast<float>(N);
        const float k = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), c);  // dx = r*u - x*k

        if (!aborted) {
            char* dxrow = dxb + static_cast<size_t>(row) * dx_pitch;
            const bool same_phase = (reinterpret_cast<uintptr_t>(dxrow) & 15) == static_cast<uintptr_t>(o);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (bits[v] == 0u) continue;
                const int idx = v * nt + tid;
                float out[VEC];
                if constexpr (PACKED) {
                    // fma(x, -k, r*u) = fma(-x, k, r*u): the product's sign is exact
                    const uint64_t nk2 = f2_pack(-k, -k);
#pragma unroll
                    for (int e = 0; e < VEC; e += 2)
                        f2_unpack(f2_fma(x2[v][e / 2], nk2, f2_mul(r2, u2[v][e / 2])), out[e], out[e + 1]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) out[e] = fmaf(-xf[v][e], k, __fmul_rn(r, uf[v][e]));
                }
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
    // one row of dgamma partials per block (zeros for a block without rows)
    if (!aborted) {
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = v * nt + tid;
            const int c0 = (16 * idx - o) / E::kBytes;
            float af[VEC];
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                if constexpr (PACKED) {
                    f2_unpack(acc2[v][e / 2], af[e], af[e + 1]);
                } else {
                    af[e] = acc[v][e];
                    af[e + 1] = acc[v][e + 1];
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if ((bits[v] >> e) & 1u) wrow[c0 + e] = af[e];
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
template <int DT, bool OFF>
static const void* ragged_pick(int pass, int vpt) {
#define RMSNORM_RG(V)                                                                        \
    case V:                                                                                  \
        return pass == 0 ? reinterpret_cast<const void*>(&fwd_ragged_kernel<DT, V, OFF>)     \
                         : reinterpret_cast<const void*>(&bwd_ragged_kernel<DT, V, OFF>);
    switch (vpt) {
        RMSNORM_RG(1)
        RMSNORM_RG(2)
        RMSNORM_RG(3)
        RMSNORM_RG(4)
        RMSNORM_RG(5)
        RMSNORM_RG(6)
    default: return nullptr;
    }
#undef RMSNORM_RG
}

const void* ragged_kernel(int pass, const Plan& p) {
    if (pass != 0 && pass != 1) return nullptr;
    switch (p.dtype) {
    case kF32: return p.offset ? ragged_pick<kF32, true>(pass, p.per_thread) : ragged_pick<kF32, false>(pass, p.per_thread);
    case kF16: return p.offset ? ragged_pick<kF16, true>(pass, p.per_thread) : ragged_pick<kF16, false>(pass, p.per_thread);
    case kBF16: return p.offset ? ragged_pick<kBF16, true>(pass, p.per_thread) : ragged_pick<kBF16, false>(pass, p.per_thread);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
