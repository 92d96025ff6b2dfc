// api.cu -- the C ABI declared in include/rmsnorm.h and include/layernorm.h:
// argument validation, launch planning (path, cluster size, threads, pipeline
// depth, persistent grid size from the device's SM count and occupancy) and
// kernel launches.
//
// Passes: 0 RMSNorm forward, 1 RMSNorm backward, 2 LayerNorm forward,
// 3 LayerNorm backward, 4 RMSNorm double backward. Passes 1, 3 and 4 are
// backward passes (two or three input row streams, per-column accumulators).
//
// Argument contract (page "Check an AI model calculation before accelerating
// it", section "The memory contract is part of the computation"): inputs are
// checked before any output is written and unsupported inputs are rejected
// rather than routed to another implementation (section "Adapting the kernel
// and moving to production": no silent fallback).
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <random>
#include <tuple>

#include "../../include/layernorm.h"
#include "../../include/rmsnorm.h"
#include "../../include/rmsnorm_double_backward.h"
#include "launch.h"
#include "tuning.h"

namespace rmsnorm {

__device__ uint32_t g_device_error;  // see rmsnorm_device_error

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSliceMaxBytes = 16384;  // widest row slice one CTA stages per tensor
// Default TMA plans, from timing grids on GB300 over row sizes 4-64 KB:
//  - every thread owns at least 2 vectors of a row (the per-row reductions,
//    barrier and square root are then amortised over >= 16 bf16 elements);
//  - the ring bytes resident per SM (stages x stage bytes x blocks) sit near
//    kRingPerSm: more requests in flight lower HBM efficiency, fewer leave it
//    latency-bound. The forward keeps 2 stages; the backward 2-4.
constexpr int kMinVpt = 2;
// Per pass (RMSNorm fwd, bwd, LayerNorm fwd, bwd, RMSNorm double backward). The
// LayerNorm forward reduces three numbers per warp per row (four butterfly sums):
// fewer warps per row and more rows in flight per SM hide that latency
// (measured: 128 threads).
constexpr int kPasses = 5;
constexpr int kThreadCap[kPasses] = {256, 128, 128, 128, 128};  // no cluster
// Row streams read per stage, reduced numbers per row, fp32 per-column planes
// staged in shared memory (gamma; the double backward's ddgamma).
constexpr int kInputs[kPasses] = {1, 2, 1, 2, 3};
constexpr int kPartials[kPasses] = {1, 1, 3, 2, 4};
constexpr int kColumnPlanes[kPasses] = {0, 1, 0, 1, 2};
// backward passes: elements a thread keeps in registers per row (x, u and the
// dgamma sums; LayerNorm also dbeta sums; the double backward x, dy and ddx)
constexpr int kMaxElemsPerThread[kPasses] = {0, 32, 0, 16, 16};
constexpr int kRingPerSm[kPasses] = {48 << 10, 96 << 10, 64 << 10, 96 << 10, 96 << 10};
constexpr int kMaxBlocksPerSm = 16;
constexpr int kRaggedFwdRingPerSm = 64 << 10;
// Rows split over a cluster pay a cluster barrier per row; more resident blocks
// hide it (up to 6 per SM for the forwards). Two stages throughout (measured,
// back to back at 512 MB per tensor: fp32 16384x8192 forward 6104 GB/s with 2
// stages against 5832 with 3, fp32 16384x16384 6273 against 5803).
constexpr int kClusterThreadCap[kPasses] = {128, 256, 128, 256, 256};
constexpr int kClusterStages[kPasses] = {2, 2, 2, 2, 2};
constexpr int kClusterBlocksPerSm[kPasses] = {6, 3, 6, 3, 3};
// Bound on each plane of the general and row-vector paths' backward workspace;
// more blocks than this add little once every SM holds a few.
constexpr int64_t kScalarWorkspaceCap = int64_t(8) << 20;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
};

struct Override {
    int threads = 0, vpt = 0, stages = 0, blocks_per_sm = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
Override g_override[kPasses];
unsigned g_override_gen = 0;
int g_row_pool = 1;  // rmsnorm_set_row_pool: 0 off, 1 on, 2 on with the forward's queue bypassed
std::atomic<unsigned> g_fwd_slot{0};  // the forward pool's next queue slot
RowPoolShape g_pool_shape;  // rmsnorm_set_row_pool_shape
std::map<std::tuple<int, int, int64_t, int, int, int, int, unsigned>, Plan> g_plans;
std::map<std::pair<const void*, int>, bool> g_attr_done;

int elem_bytes(int dt) { return dt == RMSNORM_F32 ? 4 : 2; }
int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

const void* kernel_for(int pass, const Plan& p) {
    switch (pass) {
    case 0: return fwd_kernel(p);
    case 1: return bwd_kernel(p);
    case 2: return ln_fwd_kernel(p);
    case 3: return ln_bwd_kernel(p);
    case 4: return dbwd_kernel(p);
    default: return nullptr;
    }
}

// Caller holds g_mu. The device's SM count and shared-memory limit, read once
// per device (properties of the hardware, unchanged by a device reset).
bool device_info(int dev, DeviceInfo*& out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return false;
        d.ready = true;
    }
    out = &d;
    return true;
}

// Device address of the error word in the current context, looked up on every
// call (a host-side query): an address kept from before a device reset would
// point into the destroyed context.
uint32_t* error_word_address() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<uint32_t*>(p);
}

// A ticket per backward call that uses the row pool (the owner of the queue
// word, see pool_take in bwd.cu): consecutive values of a process-wide 32-bit
// counter started at a random value, so that calls in a row never share one (a
// workspace would have to sit unused through 2^32 calls to meet its own ticket
// again).
unsigned long long next_call_ticket() {
    static std::atomic<uint32_t> counter{[] {
        const auto t = std::chrono::steady_clock::now().time_since_epoch().count();
        uint32_t seed = static_cast<uint32_t>(t) ^ static_cast<uint32_t>(t >> 32);
        try {
            std::random_device rd;  // may throw where the platform has no entropy source
            seed ^= static_cast<uint32_t>(rd());
        } catch (...) {
        }
        return seed;
    }()};
    return counter.fetch_add(1u);
}

// Caller holds g_mu. Allows the largest dynamic shared memory once per kernel and device.
bool prepare_kernel(const void* k, int dev, const DeviceInfo& di) {
    auto key = std::make_pair(k, dev);
    if (g_attr_done.count(key)) return true;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return false;
    const int dyn_max = di.smem_optin - static_cast<int>(fa.sharedSizeBytes);
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
        return false;
    if (cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return false;
    g_attr_done[key] = true;
    return true;
}

// Caller holds g_mu. Forget the attributes set on `dev`'s kernels: after a
// device reset they belong to the destroyed context and must be set again.
void forget_kernel_attributes(int dev) {
    for (auto it = g_attr_done.begin(); it != g_attr_done.end();)
        it = it->first.second == dev ? g_attr_done.erase(it) : std::next(it);
}

// Resident blocks per SM (cluster == 1) or resident clusters on the device.
bool occupancy_units(const void* k, const Plan& p, const DeviceInfo& di, int cap_per_sm, int64_t& units) {
    if (p.cluster == 1) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, p.threads + p.extra_threads, p.smem) != cudaSuccess)
            return false;
        if (cap_per_sm > 0 && n > cap_per_sm) n = cap_per_sm;
        if (n < 1) return false;
        units = static_cast<int64_t>(n) * di.sms;
        return true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.cluster * di.sms), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads + p.extra_threads), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) return false;
    if (cap_per_sm > 0) {
        const int cap = cap_per_sm * di.sms / p.cluster;
        if (n > cap) n = cap;
    }
    if (n < 1) return false;
    units = n;
    return true;
}

// TMA path: rows whose byte length is a multiple of 16, split over a cluster so
// that one CTA stages at most kSliceMaxBytes per tensor.
bool plan_tma(int pass, int64_t M, int N, int dt, int offset, int dev, const DeviceInfo& di, Plan& p) {
    const int dir = kMaxElemsPerThread[pass] > 0 ? 1 : 0;  // 0 forward, 1 backward
    const int s = elem_bytes(dt);
    const int vec = 16 / s;
    if ((static_cast<int64_t>(N) * s) % 16 != 0) return false;
    // the double backward also splits rows so that a CTA's slice fits its register
    // budget; unsplit, it may take up to kDbwdMaxThreads threads at two vectors each
    const int64_t max_cta_elems =
        pass == 4 ? static_cast<int64_t>(kMaxElemsPerThread[pass]) * kTmaMaxThreads : int64_t(1) << 30;
    const int64_t max_cta_elems_unsplit =
        pass == 4 ? static_cast<int64_t>(kMaxElemsPerThread[pass]) * kDbwdMaxThreads : max_cta_elems;
    // RMSNorm keeps rows of up to kWideRowMaxBytes in one block: the forward at 256
    // threads x 8 vectors (fp16 offset 16384x16384 forward 5847 -> 6185 GB/s against
    // the two-CTA cluster), the backward at up to kWideRowThreads threads x 4
    const int64_t max_slice_unsplit = (pass == 0 || pass == 1) ? kWideRowMaxBytes : kSliceMaxBytes;
    int cl = 1;
    while (cl <= 4 &&
           !((static_cast<int64_t>(N) * s) / cl <= (cl == 1 ? max_slice_unsplit : kSliceMaxBytes) &&
             N % (cl * vec) == 0 && N / cl <= (cl == 1 ? max_cta_elems_unsplit : max_cta_elems)))
        cl *= 2;
    if (cl > 4) return false;
    // the double backward splits rows that need four CTAs over eight: 2048-element
    // slices on 128 threads leave room for three blocks per SM, where four 256-thread
    // slices held one (fp32 16384: 5057 -> 5456 GB/s)
    if (pass == 4 && cl == 4 && N % (8 * vec) == 0) cl = 8;
    // a cluster's warps all hand one partial per row to a 32-lane read, so a
    // cluster holds at most 32 warps
    const int tmax = cl == 1 ? (pass == 4 ? kDbwdMaxThreads : (pass == 1 ? kWideRowThreads : kTmaMaxThreads))
                             : std::min(kTmaMaxThreads, 32 * 32 / cl);
    const int nvec = N / (cl * vec);
    const Override& ov = g_override[pass];
    int vpt = ov.vpt;
    if (vpt == 0) {
        const int cap = ov.threads ? ov.threads : (cl > 1 ? std::min(kClusterThreadCap[pass], tmax) : kThreadCap[pass]);
        for (vpt = kMinVpt; vpt <= 8; vpt *= 2)
            if (round_up(ceil_div(nvec, vpt), 32) <= cap) break;
        // rows wider than the thread cap holds at 8 vectors (the RMSNorm
        // backward's 16-32 KB rows): four vectors per thread on up to tmax threads
        if (vpt > 8 && !ov.threads && round_up(ceil_div(nvec, 4), 32) <= tmax) vpt = 4;
        if (vpt > 8) return false;
        if (dir == 1 && (cl == 1 || pass == 4))
            while (vpt > kMinVpt && vpt * vec > kMaxElemsPerThread[pass] &&
                   round_up(ceil_div(nvec, vpt / 2), 32) <= tmax)
                vpt /= 2;  // more threads rather than more registers
        while (vpt > 1 && ceil_div(nvec, vpt / 2) <= 32) vpt /= 2;  // tiny rows: one warp
    }
    if (vpt != 1 && vpt != 2 && vpt != 4 && vpt != 8) return false;
    int threads = ov.threads ? ov.threads : static_cast<int>(round_up(ceil_div(nvec, vpt), 32));
    if (threads < 32) threads = 32;
    // block-size bound of the kernel instance (the double backward's unsplit
    // instances of up to two vectors per thread take up to kDbwdMaxThreads)
    const int tbound = (pass == 4 && cl == 1 && vpt <= 2)   ? kDbwdMaxThreads
                       : (pass == 1 && cl == 1 && vpt <= 4) ? kWideRowThreads
                                                            : kTmaMaxThreads;
    if (threads % 32 != 0 || threads > tbound) return false;
    if (static_cast<int64_t>(threads) * vpt < nvec) return false;
    if (cl > 8 || (cl > 1 && (threads / 32) * cl > 32)) return false;
    const int slice = (N / cl) * s;
    const int stage = kInputs[pass] * slice;
    // warp partials [2][kPartials][32] floats, abort flag, fp32 per-column planes
    // of the CTA's slice; the mbarriers are counted per stage below
    const int fixed = 2 * kPartials[pass] * 32 * 4 + 16 + kColumnPlanes[pass] * (N / cl) * 4;
    // ring shape: blocks per SM and stages aiming at kRingPerSm resident per SM
    int bps = ov.blocks_per_sm;
    int stages = ov.stages;
    p.path = kPathTma;
    p.dtype = dt;
    p.offset = offset;
    p.cluster = cl;
    p.threads = threads;
    p.per_thread = vpt;
    const void* k = kernel_for(pass, p);
    if (!k || !prepare_kernel(k, dev, di)) return false;
    if (cl > 1) {
        if (!stages) stages = kClusterStages[pass];
        if (!bps) bps = kClusterBlocksPerSm[pass];
    } else if (dir == 0) {
        if (!stages) stages = 2;
        if (!bps) {
            bps = static_cast<int>(std::min<int64_t>(std::max<int64_t>(ceil_div(kRingPerSm[pass], 2 * stage), 2),
                                                     kMaxBlocksPerSm));
            // few rows per SM: the ring never reaches its steady state, and more
            // blocks put more rows in flight during the ramp (bf16 4096x4096
            // forward 16.3 -> 14.3 us with 4 blocks of 2 stages, against 3)
            if (M <= 64 * static_cast<int64_t>(di.sms) && bps < 4) bps = 4;
        }
    } else {
        if (!bps) {
            bps = static_cast<int>(std::min<int64_t>(std::max<int64_t>(kRingPerSm[pass] / (2 * stage), 1), 4));
            // few rows per SM: the ring never reaches its steady state and the
            // tail weighs more, so as many blocks as fit, up to 4 (ncu, L2 clean
            // before each kernel: bf16 8192x5120 backward row kernel 42.0 -> 35.7
            // us with 3 blocks of 2 stages instead of 2; bf16 4096x4096 19.3 ->
            // 18.1 us with 4 instead of 3; measured for the RMSNorm backward only)
            if (pass == 1 && M <= 64 * static_cast<int64_t>(di.sms)) bps = 4;
            // blocks that fit by registers alone: the ring depth is sized for those
            int fit = 0;
            p.smem = static_cast<size_t>(stage + 8) + fixed;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k, threads, p.smem) == cudaSuccess && fit >= 1 &&
                fit < bps)
                bps = fit;
        }
        if (!stages)
            stages = static_cast<int>(
                std::min<int64_t>(std::max<int64_t>(kRingPerSm[pass] / (static_cast<int64_t>(bps) * stage), 2), 4));
    }
    while (stages > 1 && static_cast<int64_t>(stages) * (stage + 8) + fixed > di.smem_optin) --stages;
    if (stages < 1) return false;
    p.stages = stages;
    p.smem = static_cast<size_t>(stages) * (stage + 8) + fixed;
    int64_t units = 0;
    if (!occupancy_units(k, p, di, bps, units)) return false;
    p.units = units < M ? units : M;
    // the RMSNorm forward and backward without clusters hand the last rows of
    // their grid out from the row pool (pool.h), when the pool kernel (one
    // producer warp more per CTA) keeps the same residency
    // (the forward's only with many rows per SM: at bf16 4096x4096 it measured
    // 16.3 -> 18.5 us; with many rows one CTA more per SM than the static plan,
    // when it fits: bf16 65536x4096 166.9 -> 165.1 us at 3 CTAs, 162.3 at 4)
    if ((pass == 1 || (pass == 0 && M > 64 * static_cast<int64_t>(di.sms))) && cl == 1 && g_row_pool &&
        stages >= 2 && stages <= kPoolMaxStages && threads <= kTmaMaxThreads && vpt <= 4 && vec * vpt < 64) {
        Plan q = p;
        q.extra_threads = 32;
        q.pool = make_row_pool(M, p.units, g_pool_shape);
        const void* kq = q.pool.head > 0 ? kernel_for(pass, q) : nullptr;
        if (kq && prepare_kernel(kq, dev, di)) {
            int64_t uq = 0;
            const int more = pass == 0 && !ov.blocks_per_sm ? bps + 1 : bps;
            if (more > bps && occupancy_units(kq, q, di, more, uq) && uq == static_cast<int64_t>(more) * di.sms &&
                uq < M) {
                q.units = uq;
                q.pool = make_row_pool(M, uq, g_pool_shape);
                if (q.pool.head > 0) p = q;
            } else if (occupancy_units(kq, q, di, bps, uq) && uq >= p.units) {
                p = q;
            }
        }
        (void)cudaGetLastError();
    }
    return true;
}

// General path: any N (<= RMSNORM_MAX_N) and element alignment, one CTA per row,
// as many resident blocks as fit.
bool plan_scalar(int pass, int64_t M, int N, int dt, int offset, int dev, const DeviceInfo& di, Plan& p) {
    const int threads = static_cast<int>(N >= kScalarThreads ? kScalarThreads : round_up(N, 32));
    p.path = kPathScalar;
    p.dtype = dt;
    p.offset = offset;
    p.cluster = 1;
    p.threads = threads;
    p.per_thread = 0;
    p.stages = 0;
    // backward: fp32 column accumulators, one plane per reduced gradient
    const int planes = (pass == 1 || pass == 4) ? 1 : (pass == 3 ? 2 : 0);
    p.smem = static_cast<size_t>(planes) * N * 4;
    const void* k = kernel_for(pass, p);
    if (!k || !prepare_kernel(k, dev, di)) return false;
    int64_t units = 0;
    if (!occupancy_units(k, p, di, 0, units)) return false;
    if (planes) {
        // keep each plane of partials (units x N floats) within kScalarWorkspaceCap
        const int64_t cap = std::max<int64_t>(di.sms, kScalarWorkspaceCap / (4 * static_cast<int64_t>(N)));
        if (units > cap) units = cap;
    }
    p.units = units < M ? units : M;
    return true;
}

// Widest aligned row (bytes) the narrow-row path takes, per pass (measured with
// the L2 flushed between runs: at exactly 2 KB the ring path is ahead for the
// RMSNorm forward, 6248 against 6102 GB/s for bf16 N = 1024, and the fp32
// RMSNorm backward, 5701 against 5390; below that, and for every other
// backward, the lanes win: bf16 N = 640 forward 5859 against 4622, bf16
// N = 1024 backward 5390 against 4099, LayerNorm by 10-60%).
int64_t lane_max_row_bytes(int pass, int dt) {
    if (pass == 0 || (pass == 1 && dt == RMSNORM_F32)) return kLaneMaxRowBytes - 16;
    return kLaneMaxRowBytes;
}

// Narrow-row path: aligned rows up to lane_max_row_bytes, a row per group of G
// lanes (the fewest, at least 4, that hold the row at up to kv_max vectors per
// lane: 4 for the forwards, 3 for the backwards, whose dgamma sums take
// registers -- bf16 N = 128 backward 5489 GB/s with 8 x 2 against 5133 with
// 4 x 4), as many blocks of kLaneThreads as fit. Overrides of threads or
// vectors per thread send the pass to the ring path instead.
bool plan_lanes(int pass, int64_t M, int N, int dt, int offset, int dev, const DeviceInfo& di, Plan& p) {
    if (pass < 0 || pass > 4) return false;
    const Override& ov = g_override[pass];
    if (ov.threads || ov.vpt) return false;
    const int64_t rowb = static_cast<int64_t>(N) * elem_bytes(dt);
    if (rowb % 16 != 0 || rowb > lane_max_row_bytes(pass, dt)) return false;
    const int nvec = static_cast<int>(rowb / 16);
    const int kv_max = (pass == 0 || pass == 2) ? 4 : (pass == 4 ? 2 : 3);
    int G = 4;
    while (G < 32 && kv_max * G < nvec) G *= 2;
    const int kv = static_cast<int>(ceil_div(nvec, G));
    if (kv < 1 || kv > 4) return false;
    p.path = kPathLanes;
    p.dtype = dt;
    p.offset = offset;
    p.cluster = 1;
    p.threads = kLaneThreads;
    p.lanes = G;
    p.per_thread = kv;
    p.stages = 0;
    const int groups = kLaneThreads / G;
    // the backwards add up their groups' sums in shared memory, a row per group
    const int64_t sums = (pass == 1 || pass == 3 || pass == 4) ? groups : 0;
    p.smem = static_cast<size_t>(sums * N * 4);
    const void* k = kernel_for(pass, p);
    if (!k || !prepare_kernel(k, dev, di)) return false;
    int64_t units = 0;
    if (!occupancy_units(k, p, di, ov.blocks_per_sm, units)) return false;
    if (sums) {
        const int64_t cap = std::max<int64_t>(di.sms, kScalarWorkspaceCap / (4 * static_cast<int64_t>(N)));
        if (units > cap) units = cap;
    }
    p.units = std::max<int64_t>(1, std::min<int64_t>(units, ceil_div(M, groups)));
    return true;
}

// Row-vector path: rows that are not 16-byte multiples or start off a 16-byte
// boundary, up to kRowVecMaxKv vectors per thread; as many blocks as fit.
bool plan_rowvec(int pass, int64_t M, int N, int dt, int offset, int dev, const DeviceInfo& di, Plan& p) {
    const int64_t rowb = static_cast<int64_t>(N) * elem_bytes(dt);
    const int64_t nvr = rowb / 16 + 2;
    const int need = static_cast<int>(ceil_div(nvr, kScalarThreads));
    int kv = 0;
    for (int cand : {1, 2, 3, 5})
        if (cand >= need) {
            kv = cand;
            break;
        }
    if (kv == 0 || kv > kRowVecMaxKv) return false;
    p.path = kPathRowVec;
    p.dtype = dt;
    p.offset = offset;
    p.cluster = 1;
    // as few threads as hold the row at kv vectors each: every warp then carries
    // the same number of vectors (514 vectors -> 192 threads x 3,
    // not 256 x 3 with one warp doing a third vector while the others wait at
    // the row barrier), and more blocks fit per SM
    p.threads = static_cast<int>(std::min<int64_t>(round_up(ceil_div(nvr, kv), 32), kScalarThreads));
    p.per_thread = kv;
    p.stages = 0;
    // per-column fp32 data in shared memory, one VEC-float slot per 16-byte
    // vector of the row's span: none (RMSNorm forward: gamma in registers), gamma
    // (the backwards), gamma and beta (LayerNorm forward)
    const int vec = 16 / elem_bytes(dt);
    const int sets[kPasses] = {0, 1, 2, 1, 0};
    p.smem = static_cast<size_t>(sets[pass]) * static_cast<size_t>(nvr) * vec * 4;
    const void* k = pass < 2 ? rowvec_kernel(pass, p) : ln_rowvec_kernel(pass, p);
    if (!k || !prepare_kernel(k, dev, di)) return false;
    int64_t units = 0;
    if (!occupancy_units(k, p, di, 0, units)) return false;
    const int planes = pass == 1 ? 1 : (pass == 3 ? 2 : 0);  // workspace planes of partials
    if (planes) {
        const int64_t cap = std::max<int64_t>(di.sms, kScalarWorkspaceCap / (4 * static_cast<int64_t>(N)));
        if (units > cap) units = cap;
    }
    // a multiple of kRowVecPhases, so that every block's rows share one 16-byte
    // phase whatever the pitch; blocks beyond the last row are idle (the
    // backward's still write a zero row of partials)
    units = std::max<int64_t>(kRowVecPhases, units / kRowVecPhases * kRowVecPhases);
    p.units = std::min<int64_t>(units, round_up(M, kRowVecPhases));
    return true;
}

// Ragged TMA path (RMSNorm and LayerNorm): rows off 16 bytes whose aligned span
// fits one ring stage of at most kSliceMaxBytes + 32 bytes; every row of a block
// shares one phase (grid a multiple of kRowVecPhases), as on the row-vector path.
bool plan_ragged(int pass, int64_t M, int N, int dt, int offset, int dev, const DeviceInfo& di, Plan& p) {
    if (pass < 0 || pass >= kPasses) return false;
    const int dir = kMaxElemsPerThread[pass] > 0 ? 1 : 0;
    // backward: elements per thread held in registers (LayerNorm: x_hat, u and
    // two accumulators per element; the double backward: x, dy, ddx and one
    // accumulator per element)
    const int max_elems = pass >= 3 ? 24 : kMaxElemsPerThread[1];
    // fp32 planes per vector slot in shared memory: none, gamma, gamma and beta,
    // gamma, gamma and ddgamma
    const int planes[kPasses] = {0, 1, 2, 1, 2};
    const int s = elem_bytes(dt);
    const int vec = 16 / s;
    const int64_t rowb = static_cast<int64_t>(N) * s;
    const int64_t stride = (rowb + 31) / 16 * 16;  // a ring stage: the widest span of any phase
    if (stride > kSliceMaxBytes + 32) return false;
    const int nslot = static_cast<int>(stride / 16);
    const Override& ov = g_override[pass];
    const int tcap = pass == 4 ? kRaggedDbwdMaxThreads : kTmaMaxThreads;
    int vpt = ov.vpt;
    int threads = ov.threads;
    if (vpt == 0 && pass == 4 && vec == 4) {
        // double backward, fp32: the fewest vectors per thread (measured: N = 4099
        // 288 x 4 at 5562 GB/s against 5171 for 224 x 5; N = 333 96 x 1 at 4504
        // against 3825 for 64 x 2)
        for (vpt = 1; vpt <= 6 && round_up(ceil_div(nslot, vpt), 32) > tcap; ++vpt) {
        }
        if (vpt > 6 || vpt * vec > max_elems) return false;
    } else if (vpt == 0 && pass == 4) {
        // double backward, 2-byte types: the fewest threads at the most vectors per
        // thread the register budget allows (measured: bf16 N = 4099 192 x 3 at 4794
        // GB/s against 4103 for 288 x 2; N = 2051 96 x 3 at 4374 against 3816 for 160 x 2)
        const int64_t t = round_up(ceil_div(nslot, max_elems / vec), 32);
        if (t > tcap) return false;
        vpt = static_cast<int>(ceil_div(nslot, t));
    } else if (vpt == 0) {
        // the fewest vectors per thread (at least two unless the row is tiny) whose
        // block fits
        for (vpt = 1; vpt <= 6; ++vpt) {
            if (vpt < 2 && nslot > 32) continue;
            if (round_up(ceil_div(nslot, vpt), 32) <= tcap) break;
        }
        if (vpt > 6 || (dir == 1 && vpt * vec > max_elems)) return false;
    }
    if (vpt < 1 || vpt > 6) return false;
    if (!threads) threads = static_cast<int>(round_up(ceil_div(nslot, vpt), 32));
    if (threads < 32 || threads % 32 != 0 || threads > tcap ||
        static_cast<int64_t>(threads) * vpt < nslot)
        return false;
    p.path = kPathRagged;
    p.dtype = dt;
    p.offset = offset;
    p.cluster = 1;
    p.threads = threads;
    p.per_thread = vpt;
    const void* k = pass < 2 ? ragged_kernel(pass, p) : (pass < 4 ? ln_ragged_kernel(pass, p) : dbwd_kernel(p));
    if (!k || !prepare_kernel(k, dev, di)) return false;
    const int64_t stage = kInputs[pass] * stride;
    const int64_t fixed =
        2 * kPartials[pass] * 32 * 4 + 16 + static_cast<int64_t>(planes[pass]) * nslot * vec * 4;
    int bps = ov.blocks_per_sm;
    int stages = ov.stages;
    if (dir == 0) {
        // the ragged forwards are latency-bound at low occupancy: a 64 KB ring per SM
        // (bf16 N = 4099: 4 blocks, 5836 GB/s at 65536 rows, against 5024 with 3)
        if (!stages) stages = 2;
        if (!bps) bps = static_cast<int>(std::min<int64_t>(std::max<int64_t>(ceil_div(kRaggedFwdRingPerSm, 2 * stage), 2),
                                                           kMaxBlocksPerSm));
    } else {
        if (!bps) {
            // the ragged backwards hold their rows in registers and are latency-bound:
            // as many blocks as fit, the ring depth shared among them (measured:
            // double backward bf16 N = 4099 2 blocks, 4794 GB/s at 65536 rows against
            // 3100 with one; fp32 N = 4099 backward 2 blocks, 5467 against 5160, and
            // LayerNorm 5257 against 4424; fp16 N = 1001 backward 6 blocks, 4390
            // against 3434 with 4)
            bps = kMaxBlocksPerSm;
            int fit = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k, threads, static_cast<size_t>(stage + 8 + fixed)) ==
                    cudaSuccess && fit >= 1 && fit < bps)
                bps = fit;
        }
        if (!stages)
            stages = static_cast<int>(
                std::min<int64_t>(std::max<int64_t>(kRingPerSm[pass] / (static_cast<int64_t>(bps) * stage), 2), 4));
    }
    while (stages > 1 && stages * (stage + 8) + fixed > di.smem_optin) --stages;
    if (stages < 1) return false;
    p.stages = stages;
    p.smem = static_cast<size_t>(stages * (stage + 8) + fixed);
    int64_t units = 0;
    if (!occupancy_units(k, p, di, bps, units)) return false;
    if (dir == 1) {
        const int64_t cap = std::max<int64_t>(di.sms, kScalarWorkspaceCap / (4 * static_cast<int64_t>(N)));
        if (units > cap) units = cap;
    }
    units = std::max<int64_t>(kRowVecPhases, units / kRowVecPhases * kRowVecPhases);
    p.units = std::min<int64_t>(units, round_up(M, kRowVecPhases));
    return true;
}

// layout: kLayoutAligned (x, y/dy/dx and gamma 16-byte aligned), kLayoutPhase
// (x and, for the backward, dy share a 16-byte phase), kLayoutMixed (anything else).
enum Layout : int { kLayoutMixed = 0, kLayoutAligned = 1, kLayoutPhase = 2 };

// Caller holds g_mu.
bool get_plan(int pass, int64_t M, int N, int dt, int offset, int layout, int dev, const DeviceInfo& di,
              Plan& p) {
    const bool tma_shape = (static_cast<int64_t>(N) * elem_bytes(dt)) % 16 == 0;
    int path = kPathScalar;
    if (layout == kLayoutAligned && tma_shape)
        path = static_cast<int64_t>(N) * elem_bytes(dt) <= lane_max_row_bytes(pass, dt) ? kPathLanes : kPathTma;
    else if (layout != kLayoutMixed) path = kPathRowVec;
    auto key = std::make_tuple(pass, dev, M, N, dt * 2 + offset, path, layout, g_override_gen);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
        p = it->second;
        return true;
    }
    bool ok = false;
    if (path == kPathLanes) {
        ok = plan_lanes(pass, M, N, dt, offset, dev, di, p);
        if (!ok) {
            (void)cudaGetLastError();
            path = kPathTma;
        }
    }
    if (path == kPathTma) ok = plan_tma(pass, M, N, dt, offset, dev, di, p);
    else if (path == kPathRowVec) {
        // the ragged TMA ring first, the row-vector kernels for wider rows
        ok = plan_ragged(pass, M, N, dt, offset, dev, di, p);
        if (!ok && pass < 4) {  // no double-backward row-vector kernel
            (void)cudaGetLastError();
            ok = plan_rowvec(pass, M, N, dt, offset, dev, di, p);
        }
    }
    if (!ok && path != kPathScalar) {
        (void)cudaGetLastError();
        path = kPathScalar;  // rows too wide for the row-vector kernels, or no TMA shape
    }
    if (path == kPathScalar) ok = plan_scalar(pass, M, N, dt, offset, dev, di, p);
    if (!ok) {
        (void)cudaGetLastError();  // leave no stale runtime error behind
        return false;
    }
    if (g_plans.size() > 4096) g_plans.clear();
    g_plans[key] = p;
    return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rmsnorm_status check_common(int64_t M, int64_t N, rmsnorm_dtype dt, int offset) {
    if (dt != RMSNORM_F32 && dt != RMSNORM_F16 && dt != RMSNORM_BF16) return RMSNORM_ERR_DTYPE;
    if (offset != 0 && offset != 1) return RMSNORM_ERR_ARG;
    if (M < 0 || M > RMSNORM_MAX_M || N < 1 || N > RMSNORM_MAX_N) return RMSNORM_ERR_SHAPE;
    return RMSNORM_OK;
}

rmsnorm_status current_device(int& dev, DeviceInfo*& di) {
    if (cudaGetDevice(&dev) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (!device_info(dev, di)) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

// The launch plan of one call, chosen under g_mu; the launches that follow run
// without the lock, so callers on different streams do not wait for each
// other's launches.
struct CallPlan {
    int dev = 0;
    Plan plan;
    uint32_t* err = nullptr;  // device error word of the current context
};

rmsnorm_status plan_call(int pass, int64_t M, int N, int dt, int offset, int layout, CallPlan& c) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo* di = nullptr;
    rmsnorm_status st = current_device(c.dev, di);
    if (st != RMSNORM_OK) return st;
    if (!get_plan(pass, M, N, dt, offset, layout, c.dev, *di, c.plan)) return RMSNORM_ERR_UNSUPPORTED;
    c.err = error_word_address();
    return c.err ? RMSNORM_OK : RMSNORM_ERR_CUDA;
}

// Launch the row kernel of `pass`. A failed launch is retried once after the
// kernel's attributes are set again: launch attributes (the opt-in shared-memory
// size) belong to a CUDA context, and a device reset since the first call on
// this device discards them while the library's record of them survives.
cudaError_t launch_pass(int pass, const CallPlan& c, const RowArgs& a, cudaStream_t s) {
    const void* k = kernel_for(pass, c.plan);
    if (!k) return cudaErrorInvalidDeviceFunction;
    cudaError_t e = launch_rows(k, c.plan, a, s);
    if (e == cudaSuccess) return e;
    (void)cudaGetLastError();
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceInfo* di = nullptr;
        int dev = 0;
        if (current_device(dev, di) != RMSNORM_OK) return cudaErrorInvalidDevice;
        forget_kernel_attributes(dev);
        if (!prepare_kernel(k, dev, *di)) return cudaErrorInvalidValue;
    }
    return launch_rows(k, c.plan, a, s);
}

}  // namespace

uint32_t* device_error_word() { return error_word_address(); }

}  // namespace rmsnorm

using namespace rmsnorm;

namespace rmsnorm {
namespace {

bool pitch_ok(int64_t ld, int64_t N, int64_t M, size_t s) {
    // ld >= N, and the whole span (M - 1) * ld + N elements addressable
    return ld >= N && ld <= (int64_t(1) << 40) / static_cast<int64_t>(s) &&
           (M <= 1 || (M - 1) <= (int64_t(1) << 46) / ld);
}

rmsnorm_status fwd_impl(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy, float* rstd, int64_t M,
                        int64_t N, float eps, rmsnorm_dtype dtype, int offset, rmsnorm_stream_t stream) {
    rmsnorm_status st = check_common(M, N, dtype, offset);
    if (st != RMSNORM_OK) return st;
    if (!std::isfinite(eps) || !(eps > 0.0f)) return RMSNORM_ERR_EPS;
    const size_t s = elem_bytes(dtype);
    if (!pitch_ok(ldx, N, M, s) || !pitch_ok(ldy, N, M, s)) return RMSNORM_ERR_SHAPE;
    if (M == 0) return RMSNORM_OK;
    if (!x || !gamma || !y || !rstd) return RMSNORM_ERR_NULL;
    if (!aligned(x, s) || !aligned(gamma, s) || !aligned(y, s) || !aligned(rstd, 4)) return RMSNORM_ERR_ALIGN;
    // TMA path: 16-byte aligned rows; otherwise the forward's row-vector path,
    // which reads x at each row's own phase and writes y at any phase
    const bool a16 = aligned(x, 16) && aligned(gamma, 16) && aligned(y, 16) && (ldx * s) % 16 == 0 &&
                     (ldy * s) % 16 == 0;
    const int layout = a16 ? kLayoutAligned : kLayoutPhase;
    CallPlan c;
    if ((st = plan_call(0, M, static_cast<int>(N), dtype, offset, layout, c)) != RMSNORM_OK) return st;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.y = y;
    a.rstd_out = rstd;
    a.M = M;
    a.N = static_cast<int>(N);
    a.ldx = ldx;
    a.ldy = ldy;
    a.eps = eps;
    a.stages = c.plan.stages;
    a.err = c.err;
    a.pool = c.plan.pool;
    if (a.pool.head > 0) {
        a.queue = fwd_queue_word(g_fwd_slot.fetch_add(1u));
        if (!a.queue) return RMSNORM_ERR_CUDA;
        a.ticket = next_call_ticket();
        a.pool_solo = g_row_pool == 2;
    }
    if (launch_pass(0, c, a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

rmsnorm_status bwd_impl(const void* dy, int64_t lddy, const void* x, int64_t ldx, const void* gamma,
                        const float* rstd, void* dx, int64_t lddx, void* dgamma, int64_t M, int64_t N,
                        rmsnorm_dtype dtype, int offset, void* workspace, size_t workspace_bytes,
                        rmsnorm_stream_t stream) {
    rmsnorm_status st = check_common(M, N, dtype, offset);
    if (st != RMSNORM_OK) return st;
    const size_t s = elem_bytes(dtype);
    if (!pitch_ok(ldx, N, M, s) || !pitch_ok(lddy, N, M, s) || !pitch_ok(lddx, N, M, s)) return RMSNORM_ERR_SHAPE;
    if (!dgamma) return RMSNORM_ERR_NULL;
    if (!aligned(dgamma, s)) return RMSNORM_ERR_ALIGN;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        if (launch_dgamma_reduce(dtype, nullptr, 0, static_cast<int>(N), workspace_pitch(N), dgamma, cs) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        return RMSNORM_OK;
    }
    if (!dy || !x || !gamma || !rstd || !dx || !workspace) return RMSNORM_ERR_NULL;
    if (!aligned(dy, s) || !aligned(x, s) || !aligned(gamma, s) || !aligned(dx, s) || !aligned(rstd, 4) ||
        !aligned(workspace, 16))
        return RMSNORM_ERR_ALIGN;
    // TMA path: 16-byte aligned rows; row-vector path: x and dy rows at the same
    // 16-byte phase (same pointer phase and pitches equal modulo 16 bytes);
    // anything else: the general path
    const bool a16 = aligned(dy, 16) && aligned(x, 16) && aligned(gamma, 16) && aligned(dx, 16) &&
                     (ldx * s) % 16 == 0 && (lddy * s) % 16 == 0 && (lddx * s) % 16 == 0;
    const bool same_phase = (reinterpret_cast<uintptr_t>(x) & 15) == (reinterpret_cast<uintptr_t>(dy) & 15) &&
                            (ldx * s) % 16 == (lddy * s) % 16;
    const int layout = a16 ? kLayoutAligned : (same_phase ? kLayoutPhase : kLayoutMixed);
    CallPlan c;
    if ((st = plan_call(1, M, static_cast<int>(N), dtype, offset, layout, c)) != RMSNORM_OK) return st;
    // a workspace too small for the row pool's partial rows but large enough for
    // one row per CTA takes the static assignment (same kernels otherwise)
    if (c.plan.pool.head > 0 && workspace_bytes < workspace_need(c.plan, N)) {
        Plan q = c.plan;
        q.pool = RowPool{};
        q.extra_threads = 0;
        if (workspace_bytes >= workspace_need(q, N)) c.plan = q;
    }
    const Plan& p = c.plan;
    if (workspace_bytes < workspace_need(p, N)) return RMSNORM_ERR_WORKSPACE;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.dy = dy;
    a.rstd_in = rstd;
    a.dx = dx;
    a.ws = static_cast<float*>(workspace);
    a.ldws = workspace_pitch(N);
    a.M = M;
    a.N = static_cast<int>(N);
    a.ldx = ldx;
    a.lddy = lddy;
    a.lddx = lddx;
    a.stages = p.stages;
    a.err = c.err;
    a.pool = p.pool;
    if (p.pool.head > 0) {
        a.queue = reinterpret_cast<unsigned long long*>(a.ws + partial_rows(p) * a.ldws);
        a.ticket = next_call_ticket();
    }
    if (launch_pass(1, c, a, cs) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (launch_dgamma_reduce(dtype, a.ws, partial_rows(p), a.N, a.ldws, dgamma, cs, nullptr, a.queue) !=
        cudaSuccess)
        return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

rmsnorm_status ln_fwd_impl(const void* x, int64_t ldx, const void* gamma, const void* beta, void* y, int64_t ldy,
                           float* mean, float* rstd, int64_t M, int64_t N, float eps, rmsnorm_dtype dtype,
                           rmsnorm_stream_t stream) {
    rmsnorm_status st = check_common(M, N, dtype, 0);
    if (st != RMSNORM_OK) return st;
    if (!std::isfinite(eps) || !(eps > 0.0f)) return RMSNORM_ERR_EPS;
    const size_t s = elem_bytes(dtype);
    if (!pitch_ok(ldx, N, M, s) || !pitch_ok(ldy, N, M, s)) return RMSNORM_ERR_SHAPE;
    if (M == 0) return RMSNORM_OK;
    if (!x || !gamma || !beta || !y) return RMSNORM_ERR_NULL;
    if (!aligned(x, s) || !aligned(gamma, s) || !aligned(beta, s) || !aligned(y, s) || !aligned(mean, 4) ||
        !aligned(rstd, 4))
        return RMSNORM_ERR_ALIGN;
    // TMA path: 16-byte aligned rows; otherwise the row-vector path (x read at
    // each row's own phase, y written at any phase)
    const bool a16 = aligned(x, 16) && aligned(gamma, 16) && aligned(beta, 16) && aligned(y, 16) &&
                     (ldx * s) % 16 == 0 && (ldy * s) % 16 == 0;
    CallPlan c;
    if ((st = plan_call(2, M, static_cast<int>(N), dtype, 0, a16 ? kLayoutAligned : kLayoutPhase, c)) !=
        RMSNORM_OK)
        return st;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.beta = beta;
    a.y = y;
    a.mean_out = mean;
    a.rstd_out = rstd;
    a.M = M;
    a.N = static_cast<int>(N);
    a.ldx = ldx;
    a.ldy = ldy;
    a.eps = eps;
    a.stages = c.plan.stages;
    a.err = c.err;
    if (launch_pass(2, c, a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

rmsnorm_status ln_bwd_impl(const void* dy, int64_t lddy, const void* x, int64_t ldx, const void* gamma,
                           const float* mean, const float* rstd, void* dx, int64_t lddx, void* dgamma, void* dbeta,
                           int64_t M, int64_t N, rmsnorm_dtype dtype, void* workspace, size_t workspace_bytes,
                           rmsnorm_stream_t stream) {
    rmsnorm_status st = check_common(M, N, dtype, 0);
    if (st != RMSNORM_OK) return st;
    const size_t s = elem_bytes(dtype);
    if (!pitch_ok(ldx, N, M, s) || !pitch_ok(lddy, N, M, s) || !pitch_ok(lddx, N, M, s)) return RMSNORM_ERR_SHAPE;
    if (!dgamma || !dbeta) return RMSNORM_ERR_NULL;
    if (!aligned(dgamma, s) || !aligned(dbeta, s)) return RMSNORM_ERR_ALIGN;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        if (launch_dgamma_reduce(dtype, nullptr, 0, static_cast<int>(N), workspace_pitch(N), dgamma, cs, dbeta) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        return RMSNORM_OK;
    }
    if (!dy || !x || !gamma || !mean || !rstd || !dx || !workspace) return RMSNORM_ERR_NULL;
    if (!aligned(dy, s) || !aligned(x, s) || !aligned(gamma, s) || !aligned(dx, s) || !aligned(mean, 4) ||
        !aligned(rstd, 4) || !aligned(workspace, 16))
        return RMSNORM_ERR_ALIGN;
    // as the RMSNorm backward: TMA path, row-vector path when x and dy rows
    // share their 16-byte phase, general path otherwise
    const bool a16 = aligned(dy, 16) && aligned(x, 16) && aligned(gamma, 16) && aligned(dx, 16) &&
                     (ldx * s) % 16 == 0 && (lddy * s) % 16 == 0 && (lddx * s) % 16 == 0;
    const bool same_phase = (reinterpret_cast<uintptr_t>(x) & 15) == (reinterpret_cast<uintptr_t>(dy) & 15) &&
                            (ldx * s) % 16 == (lddy * s) % 16;
    const int layout = a16 ? kLayoutAligned : (same_phase ? kLayoutPhase : kLayoutMixed);
    CallPlan c;
    if ((st = plan_call(3, M, static_cast<int>(N), dtype, 0, layout, c)) != RMSNORM_OK) return st;
    const Plan& p = c.plan;
    if (workspace_bytes < workspace_need(p, N, 2)) return RMSNORM_ERR_WORKSPACE;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.dy = dy;
    a.mean_in = mean;
    a.rstd_in = rstd;
    a.dx = dx;
    a.ws = static_cast<float*>(workspace);
    a.ldws = workspace_pitch(N);
    a.M = M;
    a.N = static_cast<int>(N);
    a.ldx = ldx;
    a.lddy = lddy;
    a.lddx = lddx;
    a.stages = p.stages;
    a.err = c.err;
    if (launch_pass(3, c, a, cs) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (launch_dgamma_reduce(dtype, a.ws, p.units, a.N, a.ldws, dgamma, cs, dbeta) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

rmsnorm_status bwd_bwd_impl(const void* ddx, int64_t ldddx, const void* ddgamma, const void* dy, int64_t lddy,
                            const void* x, int64_t ldx, const void* gamma, const float* rstd, void* d_dy,
                            int64_t ldd_dy, void* d_x, int64_t ldd_x, void* d_gamma, int64_t M, int64_t N,
                            rmsnorm_dtype dtype, int offset, void* workspace, size_t workspace_bytes,
                            rmsnorm_stream_t stream) {
    rmsnorm_status st = check_common(M, N, dtype, offset);
    if (st != RMSNORM_OK) return st;
    const size_t s = elem_bytes(dtype);
    if (!pitch_ok(ldddx, N, M, s) || !pitch_ok(lddy, N, M, s) || !pitch_ok(ldx, N, M, s) ||
        !pitch_ok(ldd_dy, N, M, s) || !pitch_ok(ldd_x, N, M, s))
        return RMSNORM_ERR_SHAPE;
    if (!d_gamma) return RMSNORM_ERR_NULL;
    if (!aligned(d_gamma, s)) return RMSNORM_ERR_ALIGN;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        if (launch_dgamma_reduce(dtype, nullptr, 0, static_cast<int>(N), workspace_pitch(N), d_gamma, cs) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        return RMSNORM_OK;
    }
    if (!ddx || !dy || !x || !gamma || !rstd || !d_dy || !d_x || !workspace) return RMSNORM_ERR_NULL;
    if (!aligned(ddx, s) || !aligned(ddgamma, s) || !aligned(dy, s) || !aligned(x, s) || !aligned(gamma, s) ||
        !aligned(rstd, 4) || !aligned(d_dy, s) || !aligned(d_x, s) || !aligned(workspace, 16))
        return RMSNORM_ERR_ALIGN;
    // TMA path: every row and per-column pointer 16-byte aligned with 16-byte
    // pitches; ragged TMA path: rows of x, dy and ddx at one 16-byte phase (same
    // pointer phase, pitches equal modulo 16 bytes); anything else: the general path
    const bool a16 = aligned(ddx, 16) && aligned(ddgamma, 16) && aligned(dy, 16) && aligned(x, 16) &&
                     aligned(gamma, 16) && aligned(d_dy, 16) && aligned(d_x, 16) && (ldddx * s) % 16 == 0 &&
                     (lddy * s) % 16 == 0 && (ldx * s) % 16 == 0 && (ldd_dy * s) % 16 == 0 &&
                     (ldd_x * s) % 16 == 0;
    const uintptr_t ph = reinterpret_cast<uintptr_t>(x) & 15;
    const bool same_phase = (reinterpret_cast<uintptr_t>(dy) & 15) == ph &&
                            (reinterpret_cast<uintptr_t>(ddx) & 15) == ph && (ldx * s) % 16 == (lddy * s) % 16 &&
                            (ldx * s) % 16 == (ldddx * s) % 16;
    const int layout = a16 ? kLayoutAligned : (same_phase ? kLayoutPhase : kLayoutMixed);
    CallPlan c;
    if ((st = plan_call(4, M, static_cast<int>(N), dtype, offset, layout, c)) != RMSNORM_OK) return st;
    const Plan& p = c.plan;
    const size_t need = static_cast<size_t>(p.units) * static_cast<size_t>(workspace_pitch(N)) * sizeof(float);
    if (workspace_bytes < need) return RMSNORM_ERR_WORKSPACE;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.dy = dy;
    a.rstd_in = rstd;
    a.ddx = ddx;
    a.ddg = ddgamma;
    a.d_dy = d_dy;
    a.dx = d_x;
    a.ws = static_cast<float*>(workspace);
    a.ldws = workspace_pitch(N);
    a.M = M;
    a.N = static_cast<int>(N);
    a.ldx = ldx;
    a.lddy = lddy;
    a.ldddx = ldddx;
    a.ldd_dy = ldd_dy;
    a.lddx = ldd_x;
    a.stages = p.stages;
    a.err = c.err;
    if (launch_pass(4, c, a, cs) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (launch_dgamma_reduce(dtype, a.ws, p.units, a.N, a.ldws, d_gamma, cs) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

}  // namespace
}  // namespace rmsnorm

extern "C" rmsnorm_status rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd, int64_t M,
                                      int64_t N, float eps, rmsnorm_dtype dtype, int offset,
                                      rmsnorm_stream_t stream) {
    return fwd_impl(x, N, gamma, y, N, rstd, M, N, eps, dtype, offset, stream);
}

extern "C" rmsnorm_status rmsnorm_fwd_strided(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                                              float* rstd, int64_t M, int64_t N, float eps, rmsnorm_dtype dtype,
                                              int offset, rmsnorm_stream_t stream) {
    return fwd_impl(x, ldx, gamma, y, ldy, rstd, M, N, eps, dtype, offset, stream);
}

extern "C" size_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype) {
    if (check_common(M, N, dtype, 0) != RMSNORM_OK || M == 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceInfo* di = nullptr;
    if (current_device(dev, di) != RMSNORM_OK) return 0;
    size_t need = 0;
    Plan p;
    for (int layout : {kLayoutMixed, kLayoutAligned, kLayoutPhase})
        for (int off = 0; off < 2; ++off)
            if (get_plan(1, M, static_cast<int>(N), dtype, off, layout, dev, *di, p))
                need = std::max(need, workspace_need(p, N));
    return need;
}

extern "C" rmsnorm_status rmsnorm_bwd(const void* dy, const void* x, const void* gamma, const float* rstd,
                                      void* dx, void* dgamma, int64_t M, int64_t N, rmsnorm_dtype dtype,
                                      int offset, void* workspace, size_t workspace_bytes,
                                      rmsnorm_stream_t stream) {
    return bwd_impl(dy, N, x, N, gamma, rstd, dx, N, dgamma, M, N, dtype, offset, workspace, workspace_bytes,
                    stream);
}

extern "C" rmsnorm_status rmsnorm_bwd_strided(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                                              const void* gamma, const float* rstd, void* dx, int64_t lddx,
                                              void* dgamma, int64_t M, int64_t N, rmsnorm_dtype dtype, int offset,
                                              void* workspace, size_t workspace_bytes, rmsnorm_stream_t stream) {
    return bwd_impl(dy, lddy, x, ldx, gamma, rstd, dx, lddx, dgamma, M, N, dtype, offset, workspace,
                    workspace_bytes, stream);
}

extern "C" rmsnorm_status layernorm_fwd(const void* x, int64_t ldx, const void* gamma, const void* beta, void* y,
                                        int64_t ldy, float* mean, float* rstd, int64_t M, int64_t N, float eps,
                                        rmsnorm_dtype dtype, rmsnorm_stream_t stream) {
    return ln_fwd_impl(x, ldx, gamma, beta, y, ldy, mean, rstd, M, N, eps, dtype, stream);
}

extern "C" size_t layernorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype) {
    if (check_common(M, N, dtype, 0) != RMSNORM_OK || M == 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceInfo* di = nullptr;
    if (current_device(dev, di) != RMSNORM_OK) return 0;
    size_t need = 0;
    Plan p;
    for (int layout : {kLayoutMixed, kLayoutAligned, kLayoutPhase})
        if (get_plan(3, M, static_cast<int>(N), dtype, 0, layout, dev, *di, p))
            need = std::max(need, workspace_need(p, N, 2));
    return need;
}

extern "C" rmsnorm_status layernorm_bwd(const void* dy, int64_t lddy, const void* x, int64_t ldx, const void* gamma,
                                        const float* mean, const float* rstd, void* dx, int64_t lddx, void* dgamma,
                                        void* dbeta, int64_t M, int64_t N, rmsnorm_dtype dtype, void* workspace,
                                        size_t workspace_bytes, rmsnorm_stream_t stream) {
    return ln_bwd_impl(dy, lddy, x, ldx, gamma, mean, rstd, dx, lddx, dgamma, dbeta, M, N, dtype, workspace,
                       workspace_bytes, stream);
}

extern "C" size_t rmsnorm_bwd_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype dtype) {
    if (check_common(M, N, dtype, 0) != RMSNORM_OK || M == 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceInfo* di = nullptr;
    if (current_device(dev, di) != RMSNORM_OK) return 0;
    int64_t units = 0;
    Plan p;
    for (int layout : {kLayoutMixed, kLayoutAligned, kLayoutPhase})
        for (int off = 0; off < 2; ++off)
            if (get_plan(4, M, static_cast<int>(N), dtype, off, layout, dev, *di, p) && p.units > units)
                units = p.units;
    return static_cast<size_t>(units) * static_cast<size_t>(workspace_pitch(N)) * sizeof(float);
}

extern "C" rmsnorm_status rmsnorm_bwd_bwd(const void* ddx, int64_t ldddx, const void* ddgamma, const void* dy,
                                          int64_t lddy, const void* x, int64_t ldx, const void* gamma,
                                          const float* rstd, void* d_dy, int64_t ldd_dy, void* d_x, int64_t ldd_x,
                                          void* d_gamma, int64_t M, int64_t N, rmsnorm_dtype dtype, int offset,
                                          void* workspace, size_t workspace_bytes, rmsnorm_stream_t stream) {
    return bwd_bwd_impl(ddx, ldddx, ddgamma, dy, lddy, x, ldx, gamma, rstd, d_dy, ldd_dy, d_x, ldd_x, d_gamma, M,
                        N, dtype, offset, workspace, workspace_bytes, stream);
}

extern "C" const char* rmsnorm_status_string(rmsnorm_status status) {
    switch (status) {
    case RMSNORM_OK: return "ok";
    case RMSNORM_ERR_NULL: return "a required pointer is NULL";
    case RMSNORM_ERR_SHAPE: return "M or N out of range";
    case RMSNORM_ERR_DTYPE: return "unknown dtype";
    case RMSNORM_ERR_EPS: return "eps must be finite and > 0";
    case RMSNORM_ERR_ALIGN: return "pointer not aligned as required";
    case RMSNORM_ERR_WORKSPACE: return "workspace smaller than rmsnorm_bwd_workspace_size";
    case RMSNORM_ERR_UNSUPPORTED: return "no kernel for this configuration";
    case RMSNORM_ERR_CUDA: return "CUDA runtime call or launch failed";
    case RMSNORM_ERR_ARG: return "invalid argument";
    default: return "unknown status";
    }
}

extern "C" rmsnorm_status rmsnorm_device_error(uint32_t* flags, int clear) {
    if (!flags) return RMSNORM_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (cudaMemcpyFromSymbol(flags, g_device_error, sizeof(uint32_t)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (clear) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    }
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_describe_plan(int pass, int64_t M, int64_t N, rmsnorm_dtype dtype,
                                                int aligned16, char* buf, size_t buf_len) {
    if (pass < 0 || pass >= kPasses) return RMSNORM_ERR_ARG;
    rmsnorm_status st = check_common(M, N, dtype, 0);
    if (st != RMSNORM_OK) return st;
    if (!buf || buf_len == 0) return RMSNORM_ERR_NULL;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceInfo* di = nullptr;
    if ((st = current_device(dev, di)) != RMSNORM_OK) return st;
    Plan p;
    const int layout = aligned16 == 1 ? kLayoutAligned : (aligned16 == 0 ? kLayoutPhase : kLayoutMixed);
    if (!get_plan(pass, M > 0 ? M : 1, static_cast<int>(N), dtype, 0, layout, dev, *di, p))
        return RMSNORM_ERR_UNSUPPORTED;
    char pool_text[64] = "";
    if (p.pool.head > 0)
        snprintf(pool_text, sizeof pool_text, " pool_head=%lld pool_segments=%lld", static_cast<long long>(p.pool.head),
                 static_cast<long long>(p.pool.nseg));
    if (p.path == kPathRowVec)
        snprintf(buf, buf_len, "rowvec threads=%d kv=%d units=%lld smem=%zu sms=%d", p.threads, p.per_thread,
                 static_cast<long long>(p.units), p.smem, di->sms);
    else if (p.path == kPathLanes)
        snprintf(buf, buf_len, "lanes lanes=%d kv=%d threads=%d units=%lld smem=%zu sms=%d", p.lanes, p.per_thread,
                 p.threads, static_cast<long long>(p.units), p.smem, di->sms);
    else if (p.path == kPathRagged)
        snprintf(buf, buf_len, "ragged threads=%d vpt=%d stages=%d units=%lld smem=%zu sms=%d", p.threads,
                 p.per_thread, p.stages, static_cast<long long>(p.units), p.smem, di->sms);
    else if (p.path == kPathTma)
        snprintf(buf, buf_len, "tma cluster=%d threads=%d vpt=%d stages=%d units=%lld smem=%zu sms=%d%s", p.cluster,
                 p.threads, p.per_thread, p.stages, static_cast<long long>(p.units), p.smem, di->sms, pool_text);
    else
        snprintf(buf, buf_len, "scalar threads=%d units=%lld smem=%zu sms=%d", p.threads,
                 static_cast<long long>(p.units), p.smem, di->sms);
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_set_row_pool(int enabled) {
    if (enabled < 0 || enabled > 2) return RMSNORM_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    g_row_pool = enabled;
    ++g_override_gen;
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_set_row_pool_shape(int head_pct, int head_pct_few, int len_max, int len_min) {
    if (head_pct < 0 || head_pct > 99 || head_pct_few < 0 || head_pct_few > 99 || len_max < 0 || len_min < 0 ||
        len_max > 1024 || len_min > 1024)
        return RMSNORM_ERR_ARG;
    const RowPoolShape d;
    std::lock_guard<std::mutex> lock(g_mu);
    g_pool_shape.head_pct = head_pct ? head_pct : d.head_pct;
    g_pool_shape.head_pct_few = head_pct_few ? head_pct_few : d.head_pct_few;
    g_pool_shape.len_max = len_max ? len_max : d.len_max;
    g_pool_shape.len_min = len_min ? len_min : d.len_min;
    if (g_pool_shape.len_min > g_pool_shape.len_max) g_pool_shape.len_min = g_pool_shape.len_max;
    ++g_override_gen;
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_row_pool_layout(int64_t M, int64_t G, int64_t* head, int64_t* nseg) {
    if (!head || !nseg) return RMSNORM_ERR_NULL;
    if (M < 0 || G < 1) return RMSNORM_ERR_ARG;
    const RowPool p = make_row_pool(M, G);
    *head = p.head;
    *nseg = p.nseg;
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_row_pool_segment(int64_t M, int64_t G, int64_t k, int64_t* first, int64_t* last) {
    if (!first || !last) return RMSNORM_ERR_NULL;
    if (M < 0 || G < 1) return RMSNORM_ERR_ARG;
    const RowPool p = make_row_pool(M, G);
    if (k < 0 || k >= p.nseg) return RMSNORM_ERR_ARG;
    pool_segment(p, k, *first, *last);
    return RMSNORM_OK;
}

extern "C" rmsnorm_status rmsnorm_set_launch_override(int pass, int threads, int vpt, int stages,
                                                      int blocks_per_sm) {
    if (pass < 0 || pass >= kPasses) return RMSNORM_ERR_ARG;
    if (threads < 0 || threads > 1024 || threads % 32 != 0 || stages < 0 || stages > 64 || blocks_per_sm < 0 ||
        vpt < 0 || vpt > 8)
        return RMSNORM_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    g_override[pass].threads = threads;
    g_override[pass].vpt = vpt;
    g_override[pass].stages = stages;
    g_override[pass].blocks_per_sm = blocks_per_sm;
    ++g_override_gen;
    return RMSNORM_OK;
}
