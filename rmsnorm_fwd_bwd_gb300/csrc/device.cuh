// device.cuh -- device-side building blocks shared by the RMSNorm kernels:
// element formats, 16-byte vector packing, warp reductions, and inline-PTX
// wrappers for mbarriers, TMA bulk copies (cp.async.bulk) and thread-block
// cluster distributed shared memory (sm_90+ instructions, used on sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsnorm {

// Bit 0 of the device error word: an mbarrier wait ran out of polls.
constexpr uint32_t kDevErrWaitTimeout = 1u;
// Bit 1 (debug builds, -DRMSNORM_DEBUG): a row kernel was about to read bytes
// outside the tensor it reads; the read was skipped.
constexpr uint32_t kDevErrOutOfBounds = 2u;
#ifdef RMSNORM_DEBUG
constexpr bool kDebugReads = true;
#else
constexpr bool kDebugReads = false;
#endif
// Polls of mbarrier.try_wait before a wait gives up. Each poll may suspend the
// thread for a hardware-defined interval, so this bounds a wait to well under
// a few seconds while never firing on a healthy pipeline.
constexpr uint32_t kWaitPollLimit = 1u << 21;

enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// ---------------------------------------------------------------------------
// element formats: fp32 compute, I/O in float / half / bfloat16
// ---------------------------------------------------------------------------
template <int DT> struct Elem;

template <> struct Elem<kF32> {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static float ld(const void* p, int64_t i) {
        return __ldg(static_cast<const float*>(p) + i);
    }
    __device__ __forceinline__ static void st(void* p, int64_t i, float v) {
        static_cast<float*>(p)[i] = v;
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kVec]) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[kVec]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

template <> struct Elem<kF16> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float ld(const void* p, int64_t i) {
        return __half2float(__ldg(static_cast<const __half*>(p) + i));
    }
    __device__ __forceinline__ static void st(void* p, int64_t i, float v) {
        static_cast<__half*>(p)[i] = __float2half_rn(v);
    }
    __device__ __forceinline__ static float2 word(uint32_t w) {
        __half2 h = *reinterpret_cast<const __half2*>(&w);
        return __half22float2(h);
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kVec]) {
        float2 a = word(v.x), b = word(v.y), c = word(v.z), d = word(v.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[kVec]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
};

template <> struct Elem<kBF16> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float ld(const void* p, int64_t i) {
        return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(p) + i));
    }
    __device__ __forceinline__ static void st(void* p, int64_t i, float v) {
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
    // a bfloat16 is the top half of a binary32: widening is a shift or a mask
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kVec]) {
        f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
        f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
        f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[kVec]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
};

// ---------------------------------------------------------------------------
// packed fp32 pairs: two lanes in one 64-bit register, one instruction for both
// (the f32x2 arithmetic of sm_100 and later). Each lane is rounded exactly as
// the scalar operation (fma.rn / mul.rn / add.rn per lane), so results are the
// same bits as the scalar code they replace; only the instruction count drops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {  // a * b + c, rounded once
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// y = (x * r) * g, or with the offset variant (g * x) * r where g = 1 + w (added
// here when add_one, i.e. when w arrives raw), two elements per packed
// instruction; per element the same two rounded products as the scalar form.
template <int VEC, bool OFFSET>
__device__ __forceinline__ void scale_pairs(const float (&x)[VEC], const float (&w)[VEC], bool add_one, float r,
                                            float (&o)[VEC]) {
    const uint64_t r2 = f2_pack(r, r);
#pragma unroll
    for (int e = 0; e < VEC; e += 2) {
        const uint64_t x2 = f2_pack(x[e], x[e + 1]);
        uint64_t g2 = f2_pack(w[e], w[e + 1]);
        if (add_one) g2 = f2_add(f2_pack(1.0f, 1.0f), g2);
        const uint64_t y2 = OFFSET ? f2_mul(f2_mul(g2, x2), r2) : f2_mul(f2_mul(x2, r2), g2);
        f2_unpack(y2, o[e], o[e + 1]);
    }
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
// Butterfly sum over the 32 lanes. Every lane ends with the same bits: at each
// level the two partners add the same pair of values (fp addition commutes).
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// shared memory, mbarriers, TMA bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Barrier `id` (1-15; 0 is __syncthreads) among `count` threads of the CTA, a
// multiple of 32; the other threads are not involved.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive without a transaction count (completes a phase whose count is 1).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of an mbarrier, polling at most `limit` times. On
// exhaustion sets the timeout bit in the device error word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err,
                                                  uint32_t limit = kWaitPollLimit) {
#pragma unroll 1
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicOr(err, kDevErrWaitTimeout);
    return false;
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data read back soon by another kernel (the dgamma partial rows
// the column reduce reads right after the row kernel).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte global store of four floats with an L2 cache policy.
__device__ __forceinline__ void stg_f4_hint(float* p, float a, float b, float c, float d, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d), "l"(policy)
                 : "memory");
}

// TMA bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// True when [p, p + bytes) lies in the 16-byte chunks that hold at least one
// byte of the row-major tensor at `base` (M rows of N elements of `elem` bytes,
// rows `ld` elements apart): [floor16(base), ceil16(end of the last row)). A
// copy of a row's aligned span may take the neighbouring bytes of its first
// and last chunk, never a chunk outside the tensor.
__device__ __forceinline__ bool read_in_tensor(const void* p, uint32_t bytes, const void* base, int64_t M,
                                               int64_t ld, int N, int elem) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    const uintptr_t lo = b & ~uintptr_t(15);
    const uintptr_t hi = (b + static_cast<uintptr_t>(((M - 1) * ld + N) * elem) + 15) & ~uintptr_t(15);
    const uintptr_t q = reinterpret_cast<uintptr_t>(p);
    return M > 0 && q >= lo && q + bytes <= hi;
}

// TMA bulk copy of bytes of the tensor described by (base, M, ld, N, elem). In
// debug builds the source range is checked first: outside the tensor, the copy
// is skipped and kDevErrOutOfBounds set (the stage's mbarrier then never
// completes, its bounded wait gives up and the kernel takes its abort path). In
// other builds the check compiles away.
__device__ __forceinline__ void bulk_g2s_in(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                            uint64_t policy, const void* base, int64_t M, int64_t ld, int N,
                                            int elem, uint32_t* err) {
    if (kDebugReads && !read_in_tensor(src, bytes, base, M, ld, N, elem)) {
        atomicOr(err, kDevErrOutOfBounds);
        return;
    }
    bulk_g2s(dst, src, bytes, bar, policy);
}

// ---------------------------------------------------------------------------
// thread-block clusters (a grid launched without clusters is a grid of 1-CTA
// clusters, so these read back blockIdx-like values there)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Cluster-wide barrier: every thread of every CTA in the cluster; release/acquire
// orders shared-memory writes before the barrier with reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start before the previous kernel on the stream finishes;
// griddep_wait() blocks until that kernel has completed and its memory is
// visible (a no-op when the launch did not use the attribute), so it must come
// before the first read of anything the previous kernel may have written.
// griddep_launch_dependents() lets the next such kernel begin launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asynchronous 4-byte copy global -> shared (cp.async, cached at L1), and an
// arrive on `bar` once every cp.async this thread issued so far has landed; the
// arrive does not add to the barrier's expected count (it is one of the counts
// given at init).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Arrive `count` times at once, without a transaction count.
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// 16-byte global stores: default caching, and cache-streaming (evict-first).
__device__ __forceinline__ void stg128(void* p, const uint4& v) {
    *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ void stg128_cs(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

}  // namespace rmsnorm
