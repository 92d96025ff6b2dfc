// ragged.cuh -- slot helpers of the ragged TMA kernels (ragged.cu for RMSNorm,
// ln_ragged.cu for LayerNorm): which elements of a 16-byte vector slot of a row's
// aligned span lie inside the row, and loading a slot from a ring stage with
// the other elements zeroed.
#pragma once

#include "device.cuh"

namespace rmsnorm {
namespace ragged {

// 16-byte mask keeping the elements whose bits are set in `bits` (bit e: element e).
template <int DT>
__device__ __forceinline__ uint4 keep_mask(unsigned bits) {
    uint32_t w[4];
    if (Elem<DT>::kBytes == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = ((bits >> i) & 1u) ? 0xffffffffu : 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (((bits >> (2 * i)) & 1u) ? 0x0000ffffu : 0u) | (((bits >> (2 * i + 1)) & 1u) ? 0xffff0000u : 0u);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Slot idx of a row at phase o: its elements e with column c0 + e inside [0, N).
template <int DT>
__device__ __forceinline__ unsigned slot_bits(int idx, int nv, int o, int N, int& c0) {
    constexpr int VEC = Elem<DT>::kVec;
    c0 = (16 * idx - o) / Elem<DT>::kBytes;
    unsigned bits = 0u;
    if (idx < nv) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (c0 + e >= 0 && c0 + e < N) bits |= 1u << e;
    }
    return bits;
}

// Load slot idx of a stage and zero the elements outside the row.
template <int DT>
__device__ __forceinline__ uint4 slot_load(const unsigned char* st, int idx, unsigned bits) {
    constexpr unsigned kAll = (1u << Elem<DT>::kVec) - 1u;
    if (bits == 0u) return make_uint4(0, 0, 0, 0);
    uint4 v = *reinterpret_cast<const uint4*>(st + idx * 16);
    if (bits != kAll) {
        const uint4 m = keep_mask<DT>(bits);
        v.x &= m.x; v.y &= m.y; v.z &= m.z; v.w &= m.w;
    }
    return v;
}

}  // namespace ragged
}  // namespace rmsnorm
