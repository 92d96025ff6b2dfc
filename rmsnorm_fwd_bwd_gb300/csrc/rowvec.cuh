// rowvec.cuh -- loads shared by the row-vector kernels (rowvec.cu for RMSNorm,
// ln_rowvec.cu for LayerNorm): 16-byte loads of the aligned span of a row that
// does not start on a 16-byte boundary, masked to the row and never reaching
// outside the tensor.
#pragma once

#include "device.cuh"

namespace rmsnorm {
namespace rowvec {

template <int DT> struct Raw;
template <> struct Raw<kF32> {
    __device__ __forceinline__ static uint32_t ld(const char* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }
};
template <> struct Raw<kF16> {
    __device__ __forceinline__ static uint32_t ld(const char* p) {
        return __ldg(reinterpret_cast<const unsigned short*>(p));
    }
};
template <> struct Raw<kBF16> {
    __device__ __forceinline__ static uint32_t ld(const char* p) {
        return __ldg(reinterpret_cast<const unsigned short*>(p));
    }
};

// The 16-byte vector at address A (16-byte aligned) with every element outside
// the row [rb, re) set to zero. [tb, te) is the whole tensor: a vector that
// reaches outside it is read element by element, so no byte outside the tensor
// is touched.
template <int DT>
__device__ __forceinline__ uint4 load_vec(const char* A, const char* rb, const char* re, const char* tb,
                                          const char* te) {
    using E = Elem<DT>;
    if (A >= rb && A + 16 <= re) return __ldg(reinterpret_cast<const uint4*>(A));  // wholly inside the row
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (A >= tb && A + 16 <= te) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(A));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) {
            const char* p = A + e * E::kBytes;
            if (p < rb || p >= re) {
                if (E::kBytes == 4) w[e] = 0u;
                else w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) {
        const char* p = A + e * E::kBytes;
        if (p >= rb && p < re) {
            const uint32_t v = Raw<DT>::ld(p);
            if (E::kBytes == 4) w[e] = v;
            else w[e >> 1] |= v << ((e & 1) * 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Load the vectors of one row that thread tid owns (tid, tid + nt, ...); the
// row spans (ceil16(re) - floor16(rb)) / 16 vectors, the rest are zero.
template <int DT, int KV>
__device__ __forceinline__ void load_row(const char* base, int64_t row, size_t pitch, size_t rowb, int nt,
                                         int tid, const char* tb, const char* te, uint4 (&v)[KV]) {
    const char* rb = base + static_cast<size_t>(row) * pitch;
    const char* re = rb + rowb;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(rb) & ~uintptr_t(15);
    const int nv = static_cast<int>(((reinterpret_cast<uintptr_t>(re) + 15) & ~uintptr_t(15)) - a0) / 16;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int idx = tid + k * nt;
        v[k] = idx < nv ? load_vec<DT>(reinterpret_cast<const char*>(a0) + 16 * idx, rb, re, tb, te)
                        : make_uint4(0, 0, 0, 0);
    }
}

// Minimum resident blocks passed to the forward kernels' __launch_bounds__ (0:
// none). Up to three vectors per thread the forwards fit 80 registers without
// spills when asked for three 256-thread blocks (four 192-thread blocks); left
// alone ptxas uses 100-127 (two blocks).
template <int KV> struct FwdMinBlocks { static constexpr int value = KV <= 3 ? 3 : 0; };

}  // namespace rowvec
}  // namespace rmsnorm
