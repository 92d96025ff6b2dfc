// ln_rowvec.cu -- LayerNorm forward and backward for rows that do not start on a
// 16-byte boundary (N * sizeof(dtype) not a multiple of 16, e.g. bf16 N = 4099,
// or pointers and pitches off 16 bytes), with the formulas of ln_fwd.cu and
// ln_bwd.cu.
//
// Loads as in rowvec.cu: thread t holds vectors t, t + nt, ... of the row's
// 16-byte aligned span in registers (elements outside the row masked to zero),
// the next row of the block is loaded while the current one is reduced, and
// per-column data live in shared memory at padded slots. Because a row's
// phase decides how many of its elements each warp holds, the forward counts
// them per row; its statistics take one barrier per row as in ln_fwd.cu: a
// two-pass mean and squared deviations within each warp, then the
// parallel-axis combination of the warps. The backward keeps dgamma and dbeta
// accumulators per column in shared memory and leaves one row of each per
// block in the workspace (two planes) for the fixed-order column reduce.
#include "device.cuh"
#include "launch.h"
#include "rowvec.cuh"

namespace rmsnorm {

// Minimum resident blocks passed to __launch_bounds__ (0: none). Up to three
// vectors per thread the forward fits 64 registers without spills, i.e. four
// 256-thread blocks per SM; left alone ptxas uses 80-100 (two blocks).
template <int KV> struct LnFwdRowMinBlocks { static constexpr int value = KV <= 3 ? 4 : 0; };

template <int DT, int KV>
__global__ void __launch_bounds__(kScalarThreads, (LnFwdRowMinBlocks<KV>::value))
    ln_fwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    const int padded = rowvec::pad_col(a.N) + 1;
    float* gsm = reinterpret_cast<float*>(smem);  // gamma by padded column slot
    float* bsm = gsm + padded;                    // beta by padded column slot
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
    griddep_wait();

    for (int c = tid; c < N; c += nt) {
        gsm[rowvec::pad_col(c)] = E::ld(a.gamma, c);
        bsm[rowvec::pad_col(c)] = E::ld(a.beta, c);
    }
    __syncthreads();

    const int nvr = static_cast<int>(rowb / 16) + 2;  // vectors spanned by any row
    uint4 cur[KV], nxt[KV];
    int64_t row = blockIdx.x;
    if (row < a.M) rowvec::load_row<DT, KV>(xb, row, xp, rowb, nt, tid, xb, xe, cur);
    int parity = 0;
    for (; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t next = row + gridDim.x;
        if (next < a.M) rowvec::load_row<DT, KV>(xb, next, xp, rowb, nt, tid, xb, xe, nxt);
        const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(row) * xp) & 15);

        // elements of the row this thread holds (masked ones are zero), and their sum
        float s0 = 0.f, s1 = 0.f;
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            const int c0 = (16 * idx - o) / S;
            float f[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 += f[e];
                s1 += f[e + 1];
            }
            if (idx < nvr) {
                const int lo = c0 < 0 ? 0 : c0;
                const int hi = c0 + VEC < N ? c0 + VEC : N;
                cnt += hi > lo ? hi - lo : 0;
            }
        }
        const float n_warp = warp_allsum(static_cast<float>(cnt));
        const float m_warp = n_warp > 0.f ? warp_allsum(s0 + s1) / n_warp : 0.f;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            const int c0 = (16 * idx - o) / S;
            float f[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = c0 + e;
                const float d = (idx < nvr && c >= 0 && c < N) ? f[e] - m_warp : 0.f;
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
            const int c0 = (16 * idx - o) / S;
            float f[VEC], out[VEC];
            E::unpack(cur[k], f);
            bool full = true;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = c0 + e;
                const bool in = c >= 0 && c < N;
                full = full && in;
                const int sc = rowvec::pad_col(in ? c : 0);
                out[e] = fmaf((f[e] - mu) * r, gsm[sc], bsm[sc]);
            }
            if (full && same_phase) {
                stg128(ya0 + 16 * idx, E::pack(out));
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int c = c0 + e;
                    if (c >= 0 && c < N) E::st(yrow, c, out[e]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < KV; ++k) cur[k] = nxt[k];
    }
    griddep_launch_dependents();
}

// Minimum resident blocks passed to __launch_bounds__ (0: none): left alone,
// these instances compile into 48-64 registers with spills; the fp32 ones fit
// 64 registers without spills when asked for four blocks.
template <int DT, int KV> struct LnBwdRowMinBlocks { static constexpr int value = 0; };
template <> struct LnBwdRowMinBlocks<kF32, 2> { static constexpr int value = 4; };
template <> struct LnBwdRowMinBlocks<kF32, 3> { static constexpr int value = 4; };
template <> struct LnBwdRowMinBlocks<kF16, 1> { static constexpr int value = 2; };

template <int DT, int KV>
__global__ void __launch_bounds__(kScalarThreads, (LnBwdRowMinBlocks<DT, KV>::value))
    ln_bwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    const int padded = rowvec::pad_col(a.N) + 1;
    float* gsm = reinterpret_cast<float*>(smem);  // gamma by padded column slot
    float* accg = gsm + padded;                   // dgamma accumulators
    float* accb = accg + padded;                  // dbeta accumulators
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
    griddep_wait();

    for (int c = tid; c < N; c += nt) {
        const int sc = rowvec::pad_col(c);
        gsm[sc] = E::ld(a.gamma, c);
        accg[sc] = 0.f;
        accb[sc] = 0.f;
    }
    __syncthreads();

    const int nvr = static_cast<int>(rowb / 16) + 2;
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
        const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(row) * xp) & 15);
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * nt;
            if (idx >= nvr) continue;
            const int c0 = (16 * idx - o) / S;
            float xf[VEC], df[VEC];
            E::unpack(cx[k], xf);
            E::unpack(cd[k], df);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = c0 + e;
                if (c >= 0 && c < N) {
                    const int sc = rowvec::pad_col(c);
                    const float xh = __fmul_rn(xf[e] - mu, r);
                    const float u = __fmul_rn(df[e], gsm[sc]);
                    p0 += u;
                    p1 = fmaf(u, xh, p1);
                    accg[sc] = fmaf(df[e], xh, accg[sc]);
                    accb[sc] += df[e];
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
            const int c0 = (16 * idx - o) / S;
            float xf[VEC], df[VEC], out[VEC];
            E::unpack(cx[k], xf);
            E::unpack(cd[k], df);
            bool full = true;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = c0 + e;
                const bool in = c >= 0 && c < N;
                full = full && in;
                const float xh = __fmul_rn(xf[e] - mu, r);
                const float u = __fmul_rn(df[e], gsm[rowvec::pad_col(in ? c : 0)]);
                out[e] = r * fmaf(-xh, c2, u - c1);
            }
            if (full && same_phase) {
                stg128(da0 + 16 * idx, E::pack(out));
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int c = c0 + e;
                    if (c >= 0 && c < N) E::st(dxrow, c, out[e]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            cx[k] = nx[k];
            cd[k] = nd[k];
        }
    }
    griddep_launch_dependents();
    __syncthreads();  // the last row's accumulator updates are done
    if (blockIdx.x < a.M) {
        const size_t plane = static_cast<size_t>(gridDim.x) * N;
        float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * N;
        for (int c = tid; c < N; c += nt) {
            const int sc = rowvec::pad_col(c);
            wrow[c] = accg[sc];
            wrow[plane + c] = accb[sc];
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
