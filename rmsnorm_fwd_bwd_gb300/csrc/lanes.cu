// lanes.cu -- RMSNorm and LayerNorm forward and backward, and the RMSNorm double
// backward, for narrow rows (at most 2 KB, 16-byte aligned): a row per group of G
// lanes (G = 4, 8, 16 or 32, so a group never straddles a warp; the fewest that
// hold the row at up to two to four vectors per lane), with no block barrier per
// row.
//
// The ring kernels (fwd.cu, bwd.cu, ln_fwd.cu, ln_bwd.cu) take a CTA per row and
// one barrier per row; for a row of 256 bf16 elements (32 vectors) that leaves
// one warp per CTA and few rows in flight per SM. Here each group of G lanes
// owns rows gid, gid + T, ... (T = groups in the grid), each lane KV vectors of
// a row (slots li, li + G, ...), reduced with G-lane butterflies; the rows
// that follow are loaded a few iterations ahead (RowQueue), so every lane keeps
// several rows' loads in flight. All lanes of a warp run the same number of
// iterations (that of the warp's first group) so that the butterflies always
// see the whole warp; a group past the last row computes on zeros and stores
// nothing.
//
// A lane owns the same columns in every row, so its per-column data (gamma or
// 1 + w, beta) are widened once into registers, as are the backwards' dgamma
// (and dbeta) sums; at the end the groups' sums are added in group order in
// shared memory and each block writes one row of partials for the fixed-order
// column reduce, as the other paths do.
//
// Formulas, with the I/O widened to fp32 at load: the forward of fwd.cu
// (r = 1 / sqrt(sum(x^2) / N + eps), y = (x * r) * gamma or ((1 + w) * x) * r),
// the backward of bwd.cu (u = dy * g, c = sum(u * x) / N,
// dx = r * u - x * (r^3 * c), dgamma partial += (dy * x) * r), and LayerNorm as
// in ln_fwd.cu / ln_bwd.cu (mean = sum(x) / N, var = sum((x - mean)^2) / N,
// r = 1 / sqrt(var + eps), y = x_hat * gamma + beta; dx = r * (u - mean(u) -
// x_hat * mean(u * x_hat)), dgamma += dy * x_hat, dbeta += dy).
#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

namespace {

template <int G>
__device__ __forceinline__ float group_allsum(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Row geometry shared by the kernels: group id, lane in group, warp-uniform
// iteration count.
template <int G>
struct Lanes {
    static constexpr int kGroups = kLaneThreads / G;  // row groups per block
    int li;
    int64_t gid, T, iters;
    __device__ __forceinline__ Lanes(int64_t M) {
        const int tid = threadIdx.x;
        li = tid % G;
        T = static_cast<int64_t>(gridDim.x) * kGroups;
        gid = static_cast<int64_t>(blockIdx.x) * kGroups + tid / G;
        const int64_t gid0 = static_cast<int64_t>(blockIdx.x) * kGroups + (tid & ~31) / G;
        iters = gid0 < M ? (M - 1 - gid0) / T + 1 : 0;
    }
};

// The lane's columns of a per-column vector (gamma or 1 + w, beta), widened to
// fp32 once: slots li, li + G, ... (zero past the row's end).
template <int DT, int G, int KV, bool PLUS_ONE>
__device__ __forceinline__ void load_cols(const void* src, int nvec, int li, float (&w)[KV][Elem<DT>::kVec]) {
    using E = Elem<DT>;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = li + k * G;
        E::unpack(idx < nvec ? __ldg(reinterpret_cast<const uint4*>(src) + idx) : make_uint4(0, 0, 0, 0), w[k]);
        if (PLUS_ONE) {
#pragma unroll
            for (int e = 0; e < E::kVec; ++e) w[k][e] = idx < nvec ? 1.0f + w[k][e] : 0.f;
        }
    }
}

// The lane's vectors of one row (zero past the row's end or past the last row).
template <int G, int KV>
__device__ __forceinline__ void load_row(const char* base, int64_t row, size_t pitch, int64_t M, int nvec, int li,
                                         uint4 (&v)[KV]) {
    const uint4* p = reinterpret_cast<const uint4*>(base + static_cast<size_t>(row) * pitch);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = li + k * G;
        v[k] = (row < M && idx < nvec) ? __ldg(p + idx) : make_uint4(0, 0, 0, 0);
    }
}

// Rows loaded ahead: q[0] is the current row, q[i] the row i * T after it; the
// load of the row D * T ahead is issued before the current row is reduced, so
// D + 1 rows per lane are in flight or held. Depths of 1 to 4 measured within 2%
// of each other; the deeper queue for fewer vectors per lane keeps the bytes in
// flight per lane about equal.
constexpr int lane_depth(int kv) { return kv <= 1 ? 4 : (kv == 2 ? 3 : 2); }

template <int G, int KV, int D>
struct RowQueue {
    uint4 q[D][KV];
    __device__ __forceinline__ void fill(const char* base, int64_t row, int64_t T, size_t pitch, int64_t M, int nvec,
                                         int li) {
#pragma unroll
        for (int i = 0; i < D; ++i) load_row<G, KV>(base, row + i * T, pitch, M, nvec, li, q[i]);
    }
    __device__ __forceinline__ void push(const uint4 (&v)[KV]) {
#pragma unroll
        for (int i = 0; i + 1 < D; ++i)
#pragma unroll
            for (int k = 0; k < KV; ++k) q[i][k] = q[i + 1][k];
#pragma unroll
        for (int k = 0; k < KV; ++k) q[D - 1][k] = v[k];
    }
};

template <int D>
struct ScalarQueue {
    float q[D];
    __device__ __forceinline__ void fill(const float* p, int64_t row, int64_t T, int64_t M) {
#pragma unroll
        for (int i = 0; i < D; ++i) q[i] = row + i * T < M ? __ldg(p + row + i * T) : 0.f;
    }
    __device__ __forceinline__ void push(float v) {
#pragma unroll
        for (int i = 0; i + 1 < D; ++i) q[i] = q[i + 1];
        q[D - 1] = v;
    }
};

// Sums of the block's groups, in group order, into one row of the workspace.
template <int G, int KV, int VEC>
__device__ __forceinline__ void block_partials(const float (&acc)[KV][VEC], int nvec, int N, float* red, float* wrow) {
    const int grp = threadIdx.x / G;
    const int li = threadIdx.x % G;
    float4* r4 = reinterpret_cast<float4*>(red + static_cast<size_t>(grp) * N);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = li + k * G;
        if (idx < nvec) {
#pragma unroll
            for (int q = 0; q < VEC; q += 4)
                r4[(idx * VEC + q) / 4] = make_float4(acc[k][q], acc[k][q + 1], acc[k][q + 2], acc[k][q + 3]);
        }
    }
    __syncthreads();
    for (int col = threadIdx.x; col < N; col += blockDim.x) {
        float s = 0.f;
        for (int g = 0; g < Lanes<G>::kGroups; ++g) s += red[static_cast<size_t>(g) * N + col];
        wrow[col] = s;
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// RMSNorm
// ---------------------------------------------------------------------------
template <int DT, int G, int KV, bool OFFSET>
__global__ void __launch_bounds__(kLaneThreads) fwd_lanes_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const int N = a.N;
    const int nvec = N / VEC;
    const Lanes<G> L(a.M);
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    char* yb = static_cast<char*>(a.y);

    griddep_wait();
    float g[KV][VEC];
    load_cols<DT, G, KV, OFFSET>(a.gamma, nvec, L.li, g);

    constexpr int D = lane_depth(KV);
    RowQueue<G, KV, D> xq;
    xq.fill(xb, L.gid, L.T, x_pitch, a.M, nvec, L.li);
    for (int64_t j = 0; j < L.iters; ++j) {
        const int64_t row = L.gid + j * L.T;
        uint4 nxt[KV];
        load_row<G, KV>(xb, row + D * L.T, x_pitch, a.M, nvec, L.li, nxt);
        const uint4 (&cur)[KV] = xq.q[0];
        float xf[KV][VEC];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            E::unpack(cur[k], xf[k]);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 = fmaf(xf[k][e], xf[k][e], s0);
                s1 = fmaf(xf[k][e + 1], xf[k][e + 1], s1);
            }
        }
        const float ms = group_allsum<G>(s0 + s1) / static_cast<float>(N);
        const float r = 1.0f / sqrtf(ms + a.eps);
        if (row < a.M) {
            if (L.li == 0) a.rstd_out[row] = r;
            char* yrow = yb + static_cast<size_t>(row) * y_pitch;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = L.li + k * G;
                if (idx < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = OFFSET ? (g[k][e] * xf[k][e]) * r : (xf[k][e] * r) * g[k][e];
                    stg128(yrow + idx * 16, E::pack(o));
                }
            }
        }
        xq.push(nxt);
    }
    griddep_launch_dependents();
}

template <int DT, int G, int KV, bool OFFSET>
__global__ void __launch_bounds__(kLaneThreads) bwd_lanes_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N;
    const int nvec = N / VEC;
    float* red = reinterpret_cast<float*>(smem);  // [groups][N] dgamma sums
    const Lanes<G> L(a.M);
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
    const size_t dx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    const char* dyb = static_cast<const char*>(a.dy);
    char* dxb = static_cast<char*>(a.dx);

    griddep_wait();
    float gw[KV][VEC];
    load_cols<DT, G, KV, OFFSET>(a.gamma, nvec, L.li, gw);

    float acc[KV][VEC];
#pragma unroll
    for (int k = 0; k < KV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[k][e] = 0.f;
    constexpr int D = lane_depth(KV) > 1 ? lane_depth(KV) - 1 : 1;  // two tensors per row
    RowQueue<G, KV, D> xq, dq;
    ScalarQueue<D> rq;
    xq.fill(xb, L.gid, L.T, x_pitch, a.M, nvec, L.li);
    dq.fill(dyb, L.gid, L.T, dy_pitch, a.M, nvec, L.li);
    rq.fill(a.rstd_in, L.gid, L.T, a.M);
    for (int64_t j = 0; j < L.iters; ++j) {
        const int64_t row = L.gid + j * L.T;
        const int64_t ahead = row + D * L.T;
        uint4 xn[KV], dn[KV];
        load_row<G, KV>(xb, ahead, x_pitch, a.M, nvec, L.li, xn);
        load_row<G, KV>(dyb, ahead, dy_pitch, a.M, nvec, L.li, dn);
        const float r_nxt = ahead < a.M ? __ldg(a.rstd_in + ahead) : 0.f;
        const uint4 (&xc)[KV] = xq.q[0];
        const uint4 (&dc)[KV] = dq.q[0];
        const float r = rq.q[0];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = L.li + k * G;
            if (idx < nvec) {
                float xf[VEC], df[VEC];
                E::unpack(xc[k], xf);
                E::unpack(dc[k], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float u = __fmul_rn(df[e], gw[k][e]);
                    if (e & 1) p1 = fmaf(u, xf[e], p1); else p0 = fmaf(u, xf[e], p0);
                    acc[k][e] = fmaf(__fmul_rn(df[e], xf[e]), r, acc[k][e]);
                }
            }
        }
        const float c = group_allsum<G>(p0 + p1) / static_cast<float>(N);
        const float kk = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), c);  // dx = r*u - x*kk
        if (row < a.M) {
            char* dxrow = dxb + static_cast<size_t>(row) * dx_pitch;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = L.li + k * G;
                if (idx < nvec) {
                    float xf[VEC], df[VEC], o[VEC];
                    E::unpack(xc[k], xf);
                    E::unpack(dc[k], df);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf(-xf[e], kk, __fmul_rn(r, __fmul_rn(df[e], gw[k][e])));
                    stg128(dxrow + idx * 16, E::pack(o));
                }
            }
        }
        xq.push(xn);
        dq.push(dn);
        rq.push(r_nxt);
    }
    griddep_launch_dependents();
    block_partials<G, KV, VEC>(acc, nvec, N, red, a.ws + static_cast<size_t>(blockIdx.x) * a.ldws);
}

// ---------------------------------------------------------------------------
// LayerNorm
// ---------------------------------------------------------------------------
template <int DT, int G, int KV>
__global__ void __launch_bounds__(kLaneThreads) ln_fwd_lanes_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const int N = a.N;
    const int nvec = N / VEC;
    const Lanes<G> L(a.M);
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t y_pitch = static_cast<size_t>(a.ldy) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    char* yb = static_cast<char*>(a.y);

    griddep_wait();
    float gw[KV][VEC], bw[KV][VEC];
    load_cols<DT, G, KV, false>(a.gamma, nvec, L.li, gw);
    load_cols<DT, G, KV, false>(a.beta, nvec, L.li, bw);

    constexpr int D = lane_depth(KV);
    RowQueue<G, KV, D> xq;
    xq.fill(xb, L.gid, L.T, x_pitch, a.M, nvec, L.li);
    for (int64_t j = 0; j < L.iters; ++j) {
        const int64_t row = L.gid + j * L.T;
        uint4 nxt[KV];
        load_row<G, KV>(xb, row + D * L.T, x_pitch, a.M, nvec, L.li, nxt);
        const uint4 (&cur)[KV] = xq.q[0];
        float xf[KV][VEC];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            E::unpack(cur[k], xf[k]);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 += xf[k][e];
                s1 += xf[k][e + 1];
            }
        }
        // a true division: equal elements give back their value exactly
        const float mu = group_allsum<G>(s0 + s1) / static_cast<float>(N);
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (L.li + k * G < nvec) {
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    const float d0 = xf[k][e] - mu, d1 = xf[k][e + 1] - mu;
                    q0 = fmaf(d0, d0, q0);
                    q1 = fmaf(d1, d1, q1);
                }
            }
        }
        const float var = group_allsum<G>(q0 + q1) / static_cast<float>(N);
        const float r = 1.0f / sqrtf(var + a.eps);
        if (row < a.M) {
            if (L.li == 0) {
                if (a.mean_out) a.mean_out[row] = mu;
                if (a.rstd_out) a.rstd_out[row] = r;
            }
            char* yrow = yb + static_cast<size_t>(row) * y_pitch;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = L.li + k * G;
                if (idx < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf((xf[k][e] - mu) * r, gw[k][e], bw[k][e]);
                    stg128(yrow + idx * 16, E::pack(o));
                }
            }
        }
        xq.push(nxt);
    }
    griddep_launch_dependents();
}

template <int DT, int G, int KV>
__global__ void __launch_bounds__(kLaneThreads) ln_bwd_lanes_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N;
    const int nvec = N / VEC;
    float* red = reinterpret_cast<float*>(smem);  // [groups][N] sums, dgamma then dbeta
    const Lanes<G> L(a.M);
    const size_t x_pitch = static_cast<size_t>(a.ldx) * E::kBytes;
    const size_t dy_pitch = static_cast<size_t>(a.lddy) * E::kBytes;
    const size_t dx_pitch = static_cast<size_t>(a.lddx) * E::kBytes;
    const char* xb = static_cast<const char*>(a.x);
    const char* dyb = static_cast<const char*>(a.dy);
    char* dxb = static_cast<char*>(a.dx);

    griddep_wait();
    float gw[KV][VEC];
    load_cols<DT, G, KV, false>(a.gamma, nvec, L.li, gw);

    float accg[KV][VEC], accb[KV][VEC];
#pragma unroll
    for (int k = 0; k < KV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) accg[k][e] = accb[k][e] = 0.f;
    constexpr int D = lane_depth(KV) > 1 ? lane_depth(KV) - 1 : 1;  // two tensors per row
    RowQueue<G, KV, D> xq, dq;
    ScalarQueue<D> mq, rq;
    xq.fill(xb, L.gid, L.T, x_pitch, a.M, nvec, L.li);
    dq.fill(dyb, L.gid, L.T, dy_pitch, a.M, nvec, L.li);
    mq.fill(a.mean_in, L.gid, L.T, a.M);
    rq.fill(a.rstd_in, L.gid, L.T, a.M);
    for (int64_t j = 0; j < L.iters; ++j) {
        const int64_t row = L.gid + j * L.T;
        const int64_t ahead = row + D * L.T;
        uint4 xn[KV], dn[KV];
        load_row<G, KV>(xb, ahead, x_pitch, a.M, nvec, L.li, xn);
        load_row<G, KV>(dyb, ahead, dy_pitch, a.M, nvec, L.li, dn);
        const float m_nxt = ahead < a.M ? __ldg(a.mean_in + ahead) : 0.f;
        const float r_nxt = ahead < a.M ? __ldg(a.rstd_in + ahead) : 0.f;
        const uint4 (&xc)[KV] = xq.q[0];
        const uint4 (&dc)[KV] = dq.q[0];
        const float mu = mq.q[0], r = rq.q[0];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = L.li + k * G;
            if (idx < nvec) {
                float xf[VEC], df[VEC];
                E::unpack(xc[k], xf);
                E::unpack(dc[k], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float h = __fmul_rn(xf[e] - mu, r);
                    const float u = __fmul_rn(df[e], gw[k][e]);
                    p0 += u;
                    p1 = fmaf(u, h, p1);
                    accg[k][e] = fmaf(df[e], h, accg[k][e]);
                    accb[k][e] += df[e];
                }
            }
        }
        const float c1 = group_allsum<G>(p0) / static_cast<float>(N);
        const float c2 = group_allsum<G>(p1) / static_cast<float>(N);
        if (row < a.M) {
            char* dxrow = dxb + static_cast<size_t>(row) * dx_pitch;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = L.li + k * G;
                if (idx < nvec) {
                    float xf[VEC], df[VEC], o[VEC];
                    E::unpack(xc[k], xf);
                    E::unpack(dc[k], df);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float h = __fmul_rn(xf[e] - mu, r);
                        o[e] = r * fmaf(-h, c2, __fmul_rn(df[e], gw[k][e]) - c1);
                    }
                    stg128(dxrow + idx * 16, E::pack(o));
                }
            }
        }
        xq.push(xn);
        dq.push(dn);
        mq.push(m_nxt);
        rq.push(r_nxt);
    }
    griddep_launch_dependents();
    // plane 0: dgamma partials, plane 1: dbeta partials, one row per block each
    block_partials<G, KV, VEC>(accg, nvec, N, red, a.ws + static_cast<size_t>(blockIdx.x) * a.ldws);
    __syncthreads();
    block_partials<G, KV, VEC>(accb, nvec, N, red,
                               a.ws + (static_cast<size_t>(gridDim.x) + blockIdx.x) * static_cast<size_t>(a.ldws));
}

// ---------------------------------------------------------------------------
// RMSNorm double backward (formulas of dbwd.cu): per row, with u = dy * g,
// c = mean(u * x), A = mean(ddx * x), B + D = mean(ddx * u) + mean(ddg * dy * x),
// e = ddx - r^2 * x * A: d_dy = g * r * e + r * x * ddg,
// d_x = r * ddg * dy - r^3 * (c * ddx + u * A + x * (B + D)) + 3 * r^5 * c * A * x,
// d_gamma partial += r * dy * e.
// ---------------------------------------------------------------------------
template <int DT, int G, int KV, bool OFFSET>
__global__ void __launch_bounds__(kLaneThreads) dbwd_lanes_kernel(const RowArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N;
    const int nvec = N / VEC;
    float* red = reinterpret_cast<float*>(smem);  // [groups][N] d_gamma sums
    const Lanes<G> L(a.M);
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

    griddep_wait();
    float gw[KV][VEC], qw[KV][VEC];
    load_cols<DT, G, KV, OFFSET>(a.gamma, nvec, L.li, gw);
    if (a.ddg) {
        load_cols<DT, G, KV, false>(a.ddg, nvec, L.li, qw);
    } else {
#pragma unroll
        for (int k = 0; k < KV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) qw[k][e] = 0.f;
    }
    float acc[KV][VEC];
#pragma unroll
    for (int k = 0; k < KV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[k][e] = 0.f;

    RowQueue<G, KV, 1> xq, dq, tq;
    ScalarQueue<1> rq;
    xq.fill(xb, L.gid, L.T, x_pitch, a.M, nvec, L.li);
    dq.fill(dyb, L.gid, L.T, dy_pitch, a.M, nvec, L.li);
    tq.fill(tb, L.gid, L.T, t_pitch, a.M, nvec, L.li);
    rq.fill(a.rstd_in, L.gid, L.T, a.M);
    const float inv_n = 1.0f / static_cast<float>(N);
    for (int64_t j = 0; j < L.iters; ++j) {
        const int64_t row = L.gid + j * L.T;
        const int64_t ahead = row + L.T;
        uint4 xn[KV], dn[KV], tn[KV];
        load_row<G, KV>(xb, ahead, x_pitch, a.M, nvec, L.li, xn);
        load_row<G, KV>(dyb, ahead, dy_pitch, a.M, nvec, L.li, dn);
        load_row<G, KV>(tb, ahead, t_pitch, a.M, nvec, L.li, tn);
        const float r_nxt = ahead < a.M ? __ldg(a.rstd_in + ahead) : 0.f;
        const float r = rq.q[0];
        float pc = 0.f, pa = 0.f, pb = 0.f, pd = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            if (L.li + k * G < nvec) {
                float xf[VEC], df[VEC], tf[VEC];
                E::unpack(xq.q[0][k], xf);
                E::unpack(dq.q[0][k], df);
                E::unpack(tq.q[0][k], tf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float u = __fmul_rn(df[e], gw[k][e]);
                    pc = fmaf(u, xf[e], pc);
                    pa = fmaf(tf[e], xf[e], pa);
                    pb = fmaf(tf[e], u, pb);
                    pd = fmaf(__fmul_rn(qw[k][e], df[e]), xf[e], pd);
                }
            }
        }
        const float c = group_allsum<G>(pc) * inv_n;
        const float A = group_allsum<G>(pa) * inv_n;
        const float bd = (group_allsum<G>(pb) + group_allsum<G>(pd)) * inv_n;  // B + D
        const float r2 = r * r;
        const float r3 = r2 * r;
        const float r2a = r2 * A;
        const float k5 = (3.0f * (r3 * r2)) * (c * A);
        if (row < a.M) {
            char* odx_row = odxb + static_cast<size_t>(row) * odx_pitch;
            char* ody_row = odyb + static_cast<size_t>(row) * ody_pitch;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = L.li + k * G;
                if (idx < nvec) {
                    float xf[VEC], df[VEC], tf[VEC], o_dy[VEC], o_x[VEC];
                    E::unpack(xq.q[0][k], xf);
                    E::unpack(dq.q[0][k], df);
                    E::unpack(tq.q[0][k], tf);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float x = xf[e], d = df[e], t = tf[e], g = gw[k][e], q = qw[k][e];
                        const float u = __fmul_rn(d, g);
                        const float ee = fmaf(-r2a, x, t);  // ddx - r^2 x A
                        o_dy[e] = fmaf(g * r, ee, (r * x) * q);
                        const float inner = fmaf(x, bd, fmaf(c, t, u * A));
                        o_x[e] = fmaf(k5, x, fmaf(-r3, inner, (r * q) * d));
                        acc[k][e] = fmaf(r * d, ee, acc[k][e]);
                    }
                    stg128(ody_row + idx * 16, E::pack(o_dy));
                    stg128(odx_row + idx * 16, E::pack(o_x));
                }
            }
        }
        xq.push(xn);
        dq.push(dn);
        tq.push(tn);
        rq.push(r_nxt);
    }
    griddep_launch_dependents();
    block_partials<G, KV, VEC>(acc, nvec, N, red, a.ws + static_cast<size_t>(blockIdx.x) * a.ldws);
}

// ---------------------------------------------------------------------------
// dispatch: G lanes x KV vectors, the fewest lanes (at least 4) that hold the
// row at up to kv_max vectors each: kv_max = 4 for the forwards, 3 for the
// backwards (their sums take registers), 2 for the double backward (three rows
// and two per-column vectors in registers), except where 32 lanes need more.
// Only those instances exist.
// ---------------------------------------------------------------------------
namespace {

constexpr bool lanes_instance(int pass, int G, int KV) {
    if (pass == 0 || pass == 2) return G == 4 ? KV >= 1 && KV <= 4 : KV == 3 || KV == 4;
    if (pass == 4) return G == 4 ? KV == 1 || KV == 2 : (KV == 2 || (G == 32 && (KV == 3 || KV == 4)));
    return G == 4 ? KV >= 1 && KV <= 3 : (KV == 2 || KV == 3 || (G == 32 && KV == 4));
}

template <int DT, int G, int KV>
const void* lanes_entry(int pass, bool offset) {
    if (!lanes_instance(pass, G, KV)) return nullptr;
    switch (pass) {
    case 0:
        if constexpr (lanes_instance(0, G, KV))
            return offset ? reinterpret_cast<const void*>(&fwd_lanes_kernel<DT, G, KV, true>)
                          : reinterpret_cast<const void*>(&fwd_lanes_kernel<DT, G, KV, false>);
        return nullptr;
    case 1:
        if constexpr (lanes_instance(1, G, KV))
            return offset ? reinterpret_cast<const void*>(&bwd_lanes_kernel<DT, G, KV, true>)
                          : reinterpret_cast<const void*>(&bwd_lanes_kernel<DT, G, KV, false>);
        return nullptr;
    case 2:
        if constexpr (lanes_instance(2, G, KV)) return reinterpret_cast<const void*>(&ln_fwd_lanes_kernel<DT, G, KV>);
        return nullptr;
    case 3:
        if constexpr (lanes_instance(3, G, KV)) return reinterpret_cast<const void*>(&ln_bwd_lanes_kernel<DT, G, KV>);
        return nullptr;
    case 4:
        if constexpr (lanes_instance(4, G, KV))
            return offset ? reinterpret_cast<const void*>(&dbwd_lanes_kernel<DT, G, KV, true>)
                          : reinterpret_cast<const void*>(&dbwd_lanes_kernel<DT, G, KV, false>);
        return nullptr;
    default: return nullptr;
    }
}

template <int DT, int G>
const void* lanes_kv(int pass, int KV, bool offset) {
    switch (KV) {
    case 1: return lanes_entry<DT, G, 1>(pass, offset);
    case 2: return lanes_entry<DT, G, 2>(pass, offset);
    case 3: return lanes_entry<DT, G, 3>(pass, offset);
    case 4: return lanes_entry<DT, G, 4>(pass, offset);
    default: return nullptr;
    }
}

template <int DT>
const void* lanes_pick(int pass, int G, int KV, bool offset) {
    switch (G) {
    case 4: return lanes_kv<DT, 4>(pass, KV, offset);
    case 8: return lanes_kv<DT, 8>(pass, KV, offset);
    case 16: return lanes_kv<DT, 16>(pass, KV, offset);
    case 32: return lanes_kv<DT, 32>(pass, KV, offset);
    default: return nullptr;
    }
}

}  // namespace

const void* lanes_kernel(int pass, const Plan& p) {
    switch (p.dtype) {
    case kF32: return lanes_pick<kF32>(pass, p.lanes, p.per_thread, p.offset != 0);
    case kF16: return lanes_pick<kF16>(pass, p.lanes, p.per_thread, p.offset != 0);
    case kBF16: return lanes_pick<kBF16>(pass, p.lanes, p.per_thread, p.offset != 0);
    default: return nullptr;
    }
}

}  // namespace rmsnorm
