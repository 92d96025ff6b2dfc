// rowvec.cu -- forward and backward for rows that do not start on a 16-byte
// boundary (N * sizeof(dtype) not a multiple of 16, or pointers and pitches off
// 16 bytes) and are too wide for one ring stage of the ragged TMA kernels
// (ragged.cu): rows of 16-20 KB, e.g. bf16 N = 9999. Same formulas as fwd.cu /
// bwd.cu.
//
// A row starting at byte B covers the 16-byte aligned vectors from
// floor16(B) to ceil16(B + N*s) (rows may be further apart than N elements:
// each tensor has its own row pitch). Thread t loads vectors t, t + nt, ... of that
// range with 16-byte loads; element e of vector v is column
// c = (16 v - (B mod 16)) / s + e, and elements with c outside [0, N) belong to
// the neighbouring rows and are masked to zero. A vector that would reach
// before the tensor's first byte or past its last byte is loaded element by
// element, so every access stays inside the tensor. The next row of the block
// is loaded into registers while the current one is reduced (one row of
// prefetch). The grid is a multiple of 8, so all rows of a block start at the
// same 16-byte phase and a thread owns the same columns in each of them: gamma
// (or 1 + w) sits in registers (forward) or in shared memory per vector slot
// (backward), and the backward's dgamma sums stay in registers. Outputs with the same 16-byte phase as x get 16-byte
// stores for vectors that lie wholly inside the row and element stores at the
// row's two ends (never touching a neighbour's elements); outputs with another
// phase are written element by element.
#include "device.cuh"
#include "launch.h"
#include "rowvec.cuh"

namespace rmsnorm {

template <int DT, int KV, bool OFFSET>
__global__ void __launch_bounds__(kScalarThreads, (rowvec::FwdMinBlocks<KV>::value))
    fwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    __shared__ float red[2][32];
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
    // The grid is a multiple of the number of 16-byte phases x rows cycle
    // through, so every row of this block (blockIdx.x + k * gridDim.x) starts at
    // the same phase o and each thread owns the same columns in all of them.
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * xp) & 15);
    const int nvr = static_cast<int>(rowb / 16) + 2;  // vectors spanned by any row
    griddep_wait();

    // this thread's columns of gamma (or 1 + w), in registers; 0 outside the row
    float gf[KV][VEC];
    unsigned full_mask = 0;  // bit k: vector k lies wholly inside the row
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        const int c0 = (16 * idx - o) / S;
        if (idx < nvr && c0 >= 0 && c0 + VEC <= N) full_mask |= 1u << k;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int c = c0 + e;
            const bool in = idx < nvr && c >= 0 && c < N;
            const float w = in ? E::ld(a.gamma, c) : 0.f;
            gf[k][e] = in ? (OFFSET ? 1.0f + w : w) : 0.f;
        }
    }

    uint4 cur[KV], nxt[KV];
    int64_t row = blockIdx.x;
    if (row < a.M) rowvec::load_row<DT, KV>(xb, row, xp, rowb, nt, tid, xb, xe, cur);
    int parity = 0;
    for (; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t next = row + gridDim.x;
        if (next < a.M) rowvec::load_row<DT, KV>(xb, next, xp, rowb, nt, tid, xb, xe, nxt);
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            float f[VEC];
            E::unpack(cur[k], f);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                ss0 = fmaf(f[e], f[e], ss0);  // elements outside the row were loaded as zero
                ss1 = fmaf(f[e + 1], f[e + 1], ss1);
            }
        }
        const float wsum = warp_allsum(ss0 + ss1);
        if (lane == 0) red[parity][warp] = wsum;
        __syncthreads();
        float t = lane < nwarps ? red[parity][lane] : 0.f;
        t = warp_allsum(t);
        const float r = 1.0f / sqrtf(t / static_cast<float>(N) + a.eps);
        if (tid == 0) a.rstd_out[row] = r;

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
            for (int e = 0; e < VEC; ++e) out[e] = OFFSET ? (gf[k][e] * f[e]) * r : (f[e] * r) * gf[k][e];
            if (((full_mask >> k) & 1u) && same_phase) {
                stg128(ya0 + 16 * idx, E::pack(out));
            } else {
                const int c0 = (16 * idx - o) / S;
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

template <int DT, int KV, bool OFFSET>
__global__ void __launch_bounds__(kScalarThreads) bwd_rowvec_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[2][32];
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
    // every row of this block starts at the same 16-byte phase (see the forward);
    // dy rows share it (same pointer phase, pitches equal modulo 16 bytes)
    const int o = static_cast<int>(reinterpret_cast<uintptr_t>(xb + static_cast<size_t>(blockIdx.x) * xp) & 15);
    const int nvr = static_cast<int>(rowb / 16) + 2;
    // gamma (or 1 + w) of this block's vector slots as VEC/4 planes of float4:
    // a warp reads 512 consecutive bytes per plane; 0 outside the row
    float4* gsm4 = reinterpret_cast<float4*>(smem);
    griddep_wait();
    for (int idx = tid; idx < nvr; idx += nt) {
        const int c0 = (16 * idx - o) / S;
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int c = c0 + e;
            const bool in = c >= 0 && c < N;
            const float v = in ? E::ld(a.gamma, c) : 0.f;
            w[e] = in ? (OFFSET ? 1.0f + v : v) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < VEC; q += 4) gsm4[(q / 4) * nvr + idx] = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
    }
    unsigned full_mask = 0;
    float acc[KV][VEC];
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        const int c0 = (16 * idx - o) / S;
        if (idx < nvr && c0 >= 0 && c0 + VEC <= N) full_mask |= 1u << k;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[k][e] = 0.f;
    }
    __syncthreads();

    uint4 cx[KV], cd[KV], nx[KV], nd[KV];
    int64_t row = blockIdx.x;
    if (row < a.M) {
        rowvec::load_row<DT, KV>(xb, row, xp, rowb, nt, tid, xb, xe, cx);
        rowvec::load_row<DT, KV>(db, row, dp, rowb, nt, tid, db, de, cd);
    }
    float r_next = row < a.M ? __ldg(a.rstd_in + row) : 0.f;
    int parity = 0;
    for (; row < a.M; row += gridDim.x, parity ^= 1) {
        const int64_t next = row + gridDim.x;
        const float r = r_next;
        if (next < a.M) {
            rowvec::load_row<DT, KV>(xb, next, xp, rowb, nt, tid, xb, xe, nx);
            rowvec::load_row<DT, KV>(db, next, dp, rowb, nt, tid, db, de, nd);
            r_next = __ldg(a.rstd_in + next);
        }
        // elements outside the row are zero in x and dy, and gamma is zero there
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
                    const float u = __fmul_rn(df[q + e], g[e]);
                    if (e & 1) p1 = fmaf(u, xf[q + e], p1); else p0 = fmaf(u, xf[q + e], p0);
                    acc[k][q + e] = fmaf(__fmul_rn(df[q + e], xf[q + e]), r, acc[k][q + e]);
                }
            }
        }
        const float wsum = warp_allsum(p0 + p1);
        if (lane == 0) red[parity][warp] = wsum;
        __syncthreads();
        float t = lane < nwarps ? red[parity][lane] : 0.f;
        t = warp_allsum(t);
        const float cmean = t / static_cast<float>(N);
        const float kk = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), cmean);  // dx = r*u - x*kk

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
                for (int e = 0; e < 4; ++e)
                    out[q + e] = fmaf(-xf[q + e], kk, __fmul_rn(r, __fmul_rn(df[q + e], g[e])));
            }
            if (((full_mask >> k) & 1u) && same_phase) {
                stg128(da0 + 16 * idx, E::pack(out));
            } else {
                const int c0 = (16 * idx - o) / S;
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
    // one row of dgamma partials per block (zeros for a block without rows): the
    // vector slots of one phase tile the row, so every column is written once
    float* wrow = a.ws + static_cast<size_t>(blockIdx.x) * a.ldws;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        if (idx >= nvr) continue;
        const int c0 = (16 * idx - o) / S;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int c = c0 + e;
            if (c >= 0 && c < N) wrow[c] = acc[k][e];
        }
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int DT, bool OFF>
static const void* rowvec_pick(int pass, int kv) {
#define RMSNORM_RV(K)                                                                          \
    case K:                                                                                    \
        return pass == 0 ? reinterpret_cast<const void*>(&fwd_rowvec_kernel<DT, K, OFF>)       \
                         : reinterpret_cast<const void*>(&bwd_rowvec_kernel<DT, K, OFF>);
    switch (kv) {
        RMSNORM_RV(1)
        RMSNORM_RV(2)
        RMSNORM_RV(3)
        RMSNORM_RV(5)
    default: return nullptr;
    }
#undef RMSNORM_RV
}

const void* rowvec_kernel(int pass, const Plan& p) {
    switch (p.dtype) {
    case kF32: return p.offset ? rowvec_pick<kF32, true>(pass, p.per_thread) : rowvec_pick<kF32, false>(pass, p.per_thread);
    case kF16: return p.offset ? rowvec_pick<kF16, true>(pass, p.per_thread) : rowvec_pick<kF16, false>(pass, p.per_thread);
    case kBF16: return p.offset ? rowvec_pick<kBF16, true>(pass, p.per_thread) : rowvec_pick<kBF16, false>(pass, p.per_thread);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
