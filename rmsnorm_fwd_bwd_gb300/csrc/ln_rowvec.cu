// ln_rowvec.cu -- LayerNorm forward and backward for rows that do not start on a
// 16-byte boundary (N * sizeof(dtype) not a multiple of 16, or pointers and
// pitches off 16 bytes) and are too wide for the ragged TMA kernels
// (ln_ragged.cu): rows of 16-20 KB. Formulas of ln_fwd.cu and ln_bwd.cu.
//
// Loads as in rowvec.cu: thread t holds vectors t, t + nt, ... of the row's
// 16-byte aligned span in registers (elements outside the row masked to zero),
// and the next row of the block is loaded while the current one is reduced. The
// grid is a multiple of the 16-byte phase period, so every row of a block
// starts at one phase and each thread owns the same columns in all of them:
// gamma and beta are staged once per block in shared memory by vector slot, the
// elements each warp holds are counted once, and the backward's dgamma and dbeta
// sums stay in registers (one row of each per block in the workspace, for the
// fixed-order column reduce). The forward's statistics take one barrier per row
// as in ln_fwd.cu: a two-pass mean and squared deviations within each warp, then
// the parallel-axis combination of the warps.
#include "device.cuh"
#include "launch.h"
#include "rowvec.cuh"

namespace rmsnorm {

// gamma and beta of the block's vector slots (VEC/4 float4 planes each, zero
// outside the row); every row of the block starts at 16-byte phase o
template <int DT>
__device__ __forceinline__ void stage_columns(const void* src, int N, int o, int nvr, float4* dst) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    for (int idx = threadIdx.x; idx < nvr; idx += blockDim.x) {
        const int c0 = (16 * idx - o) / E::kBytes;
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int c = c0 + e;
            w[e] = (c >= 0 && c < N) ? E::ld(src, c) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < VEC; q += 4) dst[(q / 4) * nvr + idx] = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
    }
}

template <int DT, int KV>
__global__ void __launch_bounds__(kScalarThreads, (rowvec::FwdMinBlocks<KV>::value))
    ln_fwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[2][3][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    const size_t rowb = static_cast<size_t>(N) * S;
    const size_t xp = static_cast<size_t>(a.ldx) * S;
    const size_t yp = static_cast<size_t>(a.ldy) * S;
    const char* xb = static_cast<const char*>(a.x);
    const char* xe = xb + static_cast<size_t>(a.M - 1) * xp + rowb;  // last byte of the tensor + 1
    char* yb = static_cast<char*>(a.y);
    // every row of this block (the grid is a multiple of the phase period) starts at phase o
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * xp) & 15);
    const int nvr = static_cast<int>(rowb / 16) + 2;  // vectors spanned by any row
    float4* gsm4 = reinterpret_cast<float4*>(smem);
    float4* bsm4 = gsm4 + (VEC / 4) * nvr;
    griddep_wait();
    stage_columns<DT>(a.gamma, N, o, nvr, gsm4);
    stage_columns<DT>(a.beta, N, o, nvr, bsm4);

    // elements of a row this thread and its warp hold: the same for every row here
    unsigned in_mask[KV];  // bit e of word k: element e of vector k is in the row
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        const int c0 = (16 * idx - o) / S;
        in_mask[k] = 0u;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (idx < nvr && c0 + e >= 0 && c0 + e < N) {
                in_mask[k] |= 1u << e;
                ++cnt;
            }
    }
    const float n_warp = warp_allsum(static_cast<float>(cnt));
    __syncthreads();

    uint4 cur[KV], nxt[KV];
    int64_t row = blockIdx.x;
    if (row < a.M) rowvec::load_row<DT, KV>(xb, row, xp, rowb, nt, tid, xb, xe, cur);
    int parity = 0;
    for (; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t next = row + gridDim.x;
        if (next < a.M) rowvec::load_row<DT, KV>(xb, next, xp, rowb, nt, tid, xb, xe, nxt);
        // the warp's mean (masked elements are zero), then its squared deviations
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            float f[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 += f[e];
                s1 += f[e + 1];
            }
        }
        // a true division: equal elements give back their value exactly
        const float m_warp = n_warp > 0.f ? warp_allsum(s0 + s1) / n_warp : 0.f;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            float f[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float d = ((in_mask[k] >> e) & 1u) ? f[e] - m_warp : 0.f;
                if (e & 1) q1 = fmaf(d, d, q1); else q0 = fmaf(d, d, q0);
            }
        }
        const float q_warp = warp_allsum(q0 + q1);
        if (lane == 0) {
            red[parity][0][warp] = n_warp;
            red[parity][1][warp] = m_warp;
            red[parity][2][warp] = q_warp;
        }
        __syncthreads();
        const float tn = lane < nwarps ? red[parity][0][lane] : 0.f;
        const float tm = lane < nwarps ? red[parity][1][lane] : 0.f;
        const float tq = lane < nwarps ? red[parity][2][lane] : 0.f;
        const float mu = warp_allsum(tn * tm) / static_cast<float>(N);
        const float dm = tm - mu;
        const float var = warp_allsum(fmaf(tn * dm, dm, tq)) / static_cast<float>(N);
        const float r = 1.0f / sqrtf(var + a.eps);
        if (tid == 0) {
            if (a.mean_out) a.mean_out[row] = mu;
            if (a.rstd_out) a.rstd_out[row] = r;
        }

        char* yrow = yb + static_cast<size_t>(row) * yp;
        const bool same_phase = (reinterpret_cast<uintptr_t>(yrow) & 15) == static_cast<uintptr_t>(o);
        char* ya0 = reinterpret_cast<char*>(reinterpret_cast<uintptr_t>(yrow) & ~uintptr_t(15));
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            if (idx >= nvr) continue;
            float f[VEC], out[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                const float4 g4 = gsm4[(q / 4) * nvr + idx];
                const float4 b4 = bsm4[(q / 4) * nvr + idx];
                out[q] = fmaf((f[q] - mu) * r, g4.x, b4.x);
                out[q + 1] = fmaf((f[q + 1] - mu) * r, g4.y, b4.y);
                out[q + 2] = fmaf((f[q + 2] - mu) * r, g4.z, b4.z);
                out[q + 3] = fmaf((f[q + 3] - mu) * r, g4.w, b4.w);
            }
            if (in_mask[k] == (1u << VEC) - 1u && same_phase) {
                stg128(ya0 + 16 * idx, E::pack(out));
            } else {
                const int c0 = (16 * idx - o) / S;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if ((in_mask[k] >> e) & 1u) E::st(yrow, c0 + e, out[e]);
            }
        }
#pragma unroll
        for (int k = 0; k < KV; ++k) cur[k] = nxt[k];
    }
    griddep_launch_dependents();
}

template <int DT, int KV>
__global__ void __launch_bounds__(kScalarThreads) ln_bwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[2][2][32];
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const int N = a.N;
    const size_t rowb = static_cast<size_t>(N) * S;
    const size_t xp = static_cast<size_t>(a.ldx) * S;
    const size_t dp = static_cast<size_t>(a.lddy) * S;
    const size_t op = static_cast<size_t>(a.lddx) * S;
    const char* xb = static_cast<const char*>(a.x);
    const char* xe = xb + static_cast<size_t>(a.M - 1) * xp + rowb;
    const char* db = static_cast<const char*>(a.dy);
    const char* de = db + static_cast<size_t>(a.M - 1) * dp + rowb;
    char* dxb = static_cast<char*>(a.dx);
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * xp) & 15);
    const int nvr = static_cast<int>(rowb / 16) + 2;
    float4* gsm4 = reinterpret_cast<float4*>(smem);
    griddep_wait();
    stage_columns<DT>(a.gamma, N, o, nvr, gsm4);
    unsigned in_mask[KV];
    float accg[KV][VEC], accb[KV][VEC];
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        const int c0 = (16 * idx - o) / S;
        in_mask[k] = 0u;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            if (idx < nvr && c0 + e >= 0 && c0 + e < N) in_mask[k] |= 1u << e;
            accg[k][e] = accb[k][e] = 0.f;
        }
    }
    __syncthreads();

    uint4 cx[KV], cd[KV], nx[KV], nd[KV];
    int64_t row = blockIdx.x;
    if (row < a.M) {
        rowvec::load_row<DT, KV>(xb, row, xp, rowb, nt, tid, xb, xe, cx);
        rowvec::load_row<DT, KV>(db, row, dp, rowb, nt, tid, db, de, cd);
    }
    float m_next = row < a.M ? __ldg(a.mean_in + row) : 0.f;
    float r_next = row < a.M ? __ldg(a.rstd_in + row) : 0.f;
    int parity = 0;
    for (; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t next = row + gridDim.x;
        const float mu = m_next;
        const float r = r_next;
        if (next < a.M) {
            rowvec::load_row<DT, KV>(xb, next, xp, rowb, nt, tid, xb, xe, nx);
            rowvec::load_row<DT, KV>(db, next, dp, rowb, nt, tid, db, de, nd);
            m_next = __ldg(a.mean_in + next);
            r_next = __ldg(a.rstd_in + next);
        }
        // masked elements: dy = 0 and gamma = 0, so u = 0; x_hat is masked explicitly
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            if (idx >= nvr) continue;
            float xf[VEC], df[VEC];
            E::unpack(cx[k], xf);
            E::unpack(cd[k], df);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                const float4 g4 = gsm4[(q / 4) * nvr + idx];
                const float g[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float xh = ((in_mask[k] >> (q + e)) & 1u) ? __fmul_rn(xf[q + e] - mu, r) : 0.f;
                    const float u = __fmul_rn(df[q + e], g[e]);
                    p0 += u;
                    p1 = fmaf(u, xh, p1);
                    accg[k][q + e] = fmaf(df[q + e], xh, accg[k][q + e]);
                    accb[k][q + e] += df[q + e];
                }
            }
        }
        const float w0 = warp_allsum(p0);
        const float w1 = warp_allsum(p1);
        if (lane == 0) {
            red[parity][0][warp] = w0;
            red[parity][1][warp] = w1;
        }
        __syncthreads();
        const float c1 = warp_allsum(lane < nwarps ? red[parity][0][lane] : 0.f) / static_cast<float>(N);
        const float c2 = warp_allsum(lane < nwarps ? red[parity][1][lane] : 0.f) / static_cast<float>(N);

        char* dxrow = dxb + static_cast<size_t>(row) * op;
        const bool same_phase = (reinterpret_cast<uintptr_t>(dxrow) & 15) == static_cast<uintptr_t>(o);
        char* da0 = reinterpret_cast<char*>(reinterpret_cast<uintptr_t>(dxrow) & ~uintptr_t(15));
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            if (idx >= nvr) continue;
            float xf[VEC], df[VEC], out[VEC];
            E::unpack(cx[k], xf);
            E::unpack(cd[k], df);
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                const float4 g4 = gsm4[(q / 4) * nvr + idx];
                const float g[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float xh = __fmul_rn(xf[q + e] - mu, r);
                    const float u = __fmul_rn(df[q + e], g[e]);
                    out[q + e] = r * fmaf(-xh, c2, u - c1);
                }
            }
            if (in_mask[k] == (1u << VEC) - 1u && same_phase) {
                stg128(da0 + 16 * idx, E::pack(out));
            } else {
                const int c0 = (16 * idx - o) / S;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if ((in_mask[k] >> e) & 1u) E::st(dxrow, c0 + e, out[e]);
            }
        }
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            cx[k] = nx[k];
            cd[k] = nd[k];
        }
    }
    griddep_launch_dependents();
    // one row of dgamma partials (plane 0) and dbeta partials (plane 1) per block,
    // zeros for a block without rows; the vector slots tile the row
    const size_t plane = static_cast<size_t>(gridDim.x) * a.ldws;
    float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        if (idx >= nvr) continue;
        const int c0 = (16 * idx - o) / S;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if ((in_mask[k] >> e) & 1u) {
                wrow[c0 + e] = accg[k][e];
                wrow[plane + c0 + e] = accb[k][e];
            }
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT>
static const void* ln_rowvec_pick(int pass, int kv) {
#define LAYERNORM_RV(K)                                                                   \
    case K:                                                                               \
        return pass == 2 ? reinterpret_cast<const void*>(&ln_fwd_rowvec_kernel<DT, K>)    \
                         : reinterpret_cast<const void*>(&ln_bwd_rowvec_kernel<DT, K>);
    switch (kv) {
        LAYERNORM_RV(1)
        LAYERNORM_RV(2)
        LAYERNORM_RV(3)
        LAYERNORM_RV(5)
    default: return nullptr;
    }
#undef LAYERNORM_RV
}

const void* ln_rowvec_kernel(int pass, const Plan& p) {
    switch (p.dtype) {
    case kF32: return ln_rowvec_pick<kF32>(pass, p.per_thread);
    case kF16: return ln_rowvec_pick<kF16>(pass, p.per_thread);
    case kBF16: return ln_rowvec_pick<kBF16>(pass, p.per_thread);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
