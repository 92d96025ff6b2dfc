// pool.h -- the backward's row pool: how the rows of a persistent grid are split
// into per-CTA heads and a queue of segments, shared by the planner (host) and the
// backward row kernel (device). Internal: not part of the public ABI.
//
// With a static assignment (CTA b takes rows b, b + G, b + 2G, ...) the CTAs of a
// persistent grid finish far apart: under a full HBM stream some SMs are served
// more slowly than others (measured on GB300 with a backward-shaped TMA stream,
// 65536 rows of 8 KB read twice and written once: CTA end times spread over
// 56-70 us of a 250 us kernel; 226-230 us in all once rows are handed out
// dynamically, one at a time). The pool keeps the fixed assignment for most rows
// and hands the rest out dynamically, in a way that leaves dgamma independent of
// who ran what:
//
//   * CTA b first takes `head` rows of its own, rows b + j * G for j < head, and
//     sums their dgamma terms into partial row b;
//   * the remaining rows [G * head, M) are cut into segments of consecutive rows
//     in up to three tiers of decreasing length (long segments first, short ones
//     at the end, where the last CTAs to finish decide the kernel's time), and the
//     CTAs take segments from an atomic queue until it is empty. Segment k's terms
//     are summed, in row order, into partial row G + k.
//
// Every partial row therefore covers a fixed set of rows summed in a fixed order,
// and the column reduce adds the G + nseg partial rows in a fixed order: dgamma
// is bitwise reproducible however the queue hands out the segments.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define RMSNORM_HOST_DEVICE __host__ __device__
#else
#define RMSNORM_HOST_DEVICE
#endif

namespace rmsnorm {

constexpr int kPoolTiers = 3;

// The queue word after a call: the column reduce that follows the row kernel
// stores this (a count no call can reach), so that the next call -- even a replay
// of a captured CUDA graph, which repeats the same ticket -- opens a fresh queue.
constexpr unsigned long long kPoolClosed = 0xffffffffull;

struct RowPool {
    int64_t head = 0;                     // rows per CTA taken before the queue; 0: no pool
    int64_t nseg = 0;                     // segments in the queue
    int64_t row0[kPoolTiers] = {};        // first row of each tier
    int64_t rows_end[kPoolTiers] = {};    // one past the last row of each tier
    int64_t seg0[kPoolTiers + 1] = {};    // first segment of each tier; seg0[kPoolTiers] = nseg
    int len[kPoolTiers] = {};             // rows per segment in each tier (a tier's last may be shorter)
};

// Rows [first, last) of segment k, 0 <= k < nseg.
RMSNORM_HOST_DEVICE inline void pool_segment(const RowPool& p, int64_t k, int64_t& first, int64_t& last) {
    int t = 0;
    while (t + 1 < kPoolTiers && k >= p.seg0[t + 1]) ++t;
    first = p.row0[t] + (k - p.seg0[t]) * p.len[t];
    last = first + p.len[t];
    if (last > p.rows_end[t]) last = p.rows_end[t];
}

// The pool for M rows over G CTAs; head = 0 (no pool: the static assignment)
// when there are fewer than 4 rows per CTA. Heads take 90% of the rows (92% below
// 64 rows per CTA); the rest go to the queue: 60% in segments of R/8 rows
// (4-16), 25% in half that length, 15% in a quarter of it (at least 4 rows).
// Measured backward (row kernel + column reduce, L2 evict-last partial rows),
// static -> pool: bf16 65536x4096 250.2 -> 242.5 us, bf16 32768x4096 132.4 ->
// 127.8, fp16 16384x8192 138.9 -> 131.7; heads of 80-88% and segments of at
// most 8 or up to 32 rows measured 0.5-5 us slower at one or more of these.
// The shape knobs (percent of rows in the heads at >= 64 and < 64 rows per CTA;
// longest and shortest segment) exist for tuning; RowPoolShape{} is the default.
struct RowPoolShape {
    int head_pct = 90, head_pct_few = 92, len_max = 16, len_min = 4;
};

inline RowPool make_row_pool(int64_t M, int64_t G, const RowPoolShape& sh = RowPoolShape{}) {
    RowPool p;
    if (G <= 0 || M < 4 * G) return p;
    const int64_t R = M / G;
    const int64_t head = (R >= 64 ? M * sh.head_pct / 100 : M * sh.head_pct_few / 100) / G;
    if (head < 1 || G * head >= M) return p;
    const int64_t pool0 = G * head;
    const int64_t rows = M - pool0;
    int l1 = static_cast<int>(R / 8);
    l1 = l1 < sh.len_min ? sh.len_min : (l1 > sh.len_max ? sh.len_max : l1);
    const int l2 = l1 / 2 < sh.len_min ? sh.len_min : l1 / 2;
    const int l3 = l1 / 4 < sh.len_min ? sh.len_min : l1 / 4;
    const int64_t n1 = rows * 60 / 100, n2 = rows * 25 / 100;
    const int64_t tier_rows[kPoolTiers] = {n1, n2, rows - n1 - n2};
    const int lens[kPoolTiers] = {l1, l2, l3};
    int64_t at = pool0, seg = 0;
    for (int t = 0; t < kPoolTiers; ++t) {
        p.row0[t] = at;
        at += tier_rows[t];
        p.rows_end[t] = at;
        p.len[t] = lens[t];
        p.seg0[t] = seg;
        seg += (tier_rows[t] + lens[t] - 1) / lens[t];
    }
    p.seg0[kPoolTiers] = seg;
    p.nseg = seg;
    p.head = head;
    return p;
}

}  // namespace rmsnorm
