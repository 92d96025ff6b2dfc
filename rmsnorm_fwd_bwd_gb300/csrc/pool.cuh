// pool.cuh -- device side of the row pool (pool.h) for the RMSNorm backward,
// whose partial rows need the call's queue to be exact: the queue word protocol,
// and the row sequence one CTA's producer lane walks through. Internal.
#pragma once

#include "device.cuh"
#include "launch.h"

namespace rmsnorm {

// The pool's queue word holds {ticket (high 32 bits), segments taken (low 32)}.
// It is this call's when it carries the call's ticket and a count of at most
// nseg + 2G (a CTA stops after its first take past the end, and makes at most one
// extra take while the word is being opened); anything else -- a word left by an
// earlier call, never written, or holding another tensor's bytes -- is not.
__device__ __forceinline__ bool pool_word_ours(unsigned long long w, uint32_t ticket, int64_t nseg, int64_t G) {
    return (w >> 32) == ticket && static_cast<int64_t>(w & 0xffffffffull) <= nseg + 2 * G;
}

// CTA 0, at the start: make the word this call's with no segment taken (one
// compare-and-swap from whatever it holds to {ticket, 0}; bounded retries).
__device__ __forceinline__ void pool_open(unsigned long long* q, uint32_t ticket, int64_t nseg, int64_t G,
                                          uint32_t* err) {
    const unsigned long long mine = static_cast<unsigned long long>(ticket) << 32;
    unsigned long long w = __ldcg(q);
#pragma unroll 1
    for (uint32_t i = 0; i < kWaitPollLimit; ++i) {
        if (pool_word_ours(w, ticket, nseg, G)) return;
        const unsigned long long prev = atomicCAS(q, w, mine);
        if (prev == w) return;
        w = prev;
    }
    atomicOr(err, kDevErrWaitTimeout);
}

// The segment a take got, from the value `old` its fetch-and-add returned; -1
// when the queue is empty. Takes are single fetch-and-adds, issued ahead of need
// so that their round trip overlaps rows still in the ring (a compare-and-swap
// loop here serialises the CTAs that take at once). An add that found the word
// not yet this call's (CTA 0 had not opened it) opens it itself, taking segment
// 0, or adds again once another CTA has; bounded, and on exhaustion the timeout
// bit is set and the CTA takes no more segments (the others still empty the queue).
__device__ __forceinline__ int64_t pool_segment_of(unsigned long long old, unsigned long long* q, uint32_t ticket,
                                                   int64_t nseg, int64_t G, uint32_t* err) {
    if (pool_word_ours(old, ticket, nseg, G)) {
        const int64_t k = static_cast<int64_t>(old & 0xffffffffull);
        return k < nseg ? k : -1;
    }
    const unsigned long long mine = static_cast<unsigned long long>(ticket) << 32;
    unsigned long long w = old + 1;  // the word after this CTA's add, unless others added too
#pragma unroll 1
    for (uint32_t i = 0; i < kWaitPollLimit; ++i) {
        const unsigned long long prev = atomicCAS(q, w, mine | 1ull);
        if (prev == w) return 0;
        if (pool_word_ours(prev, ticket, nseg, G)) {
            const int64_t k = static_cast<int64_t>(atomicAdd(q, 1ull) & 0xffffffffull);
            return k < nseg ? k : -1;
        }
        w = prev;
    }
    atomicOr(err, kDevErrWaitTimeout);
    return -1;
}

// Bounded wait on an mbarrier phase that also gives up as soon as `abort` is
// set (by a thread whose own wait gave up); sets the timeout bit on exhaustion.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, uint32_t* err,
                                                   volatile int* abort) {
#pragma unroll 1
    for (uint32_t i = 0; i < kWaitPollLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    atomicOr(err, kDevErrWaitTimeout);
    return false;
}

// The rows of one CTA, in the order its producer issues them: the head rows
// b + j * G (j < pool.head; partial row b after the last), then the rows of each
// segment taken from the queue (partial row G + k after segment k's last row).
// A take is a fetch-and-add issued kPoolTakeAhead rows before its result is
// needed, so its round trip overlaps rows already in the ring.
struct PoolRows {
    int64_t heads = 0, seg_row = 0, seg_end = 0, seg_id = -1;  // seg_id -2: queue empty
    unsigned long long pend = 0;
    bool pend_on = false;

    __device__ __forceinline__ void take_ahead(const RowArgs& a) {
        if (!pend_on) {
            pend = atomicAdd(a.queue, 1ull);
            pend_on = true;
        }
    }
    // The next row (-1: none left) and in `unit` the partial row to write after
    // it (-1: none).
    __device__ __forceinline__ int64_t next(const RowArgs& a, int64_t G, uint32_t ticket, int64_t& unit) {
        int64_t row = -1;
        unit = -1;
        if (heads < a.pool.head) {
            row = static_cast<int64_t>(blockIdx.x) + heads * G;
            if (++heads == a.pool.head) unit = blockIdx.x;
            if (a.pool.head - heads <= kPoolTakeAhead) take_ahead(a);
        } else if (seg_id != -2) {
            if (seg_row >= seg_end) {
                take_ahead(a);
                pend_on = false;
                const int64_t k = pool_segment_of(pend, a.queue, ticket, a.pool.nseg, G, a.err);
                if (k >= 0) pool_segment(a.pool, k, seg_row, seg_end);
                seg_id = k >= 0 ? k : -2;
            }
            if (seg_id >= 0) {
                row = seg_row++;
                if (seg_row == seg_end) unit = G + seg_id;
                if (seg_end - seg_row <= kPoolTakeAhead) take_ahead(a);
            }
        }
        return row;
    }
};

}  // namespace rmsnorm
