/*
 * tuning.h -- internal tuning hook of librmsnorm.so; not part of the public
 * boundary in include/. Used by the tests and the benchmark to force a launch
 * shape when comparing plans.
 */
#pragma once

#include "../../include/rmsnorm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Override the TMA-path launch shape for one pass (0 = forward, 1 = backward,
 * 2 / 3 = LayerNorm forward / backward, 4 = double backward). threads: threads
 * per block (multiple of 32); vpt: 16-byte vectors per thread (1 to 8; the
 * aligned TMA path takes 1, 2, 4 or 8, the ragged one 1 to 6); stages:
 * pipeline depth; blocks_per_sm: cap on resident blocks per SM. Any value 0
 * keeps the built-in choice; all zeros restores the defaults. A shape that
 * cannot hold the row makes the following calls fail with
 * RMSNORM_ERR_UNSUPPORTED. Process-wide: it changes the plans of every later
 * call, from any thread, until it is reset.
 */
rmsnorm_status rmsnorm_set_launch_override(int pass, int threads, int vpt, int stages,
                                           int blocks_per_sm);

/*
 * Turn the RMSNorm forward's and backward's row pool on (1, the default) or off
 * (0: every CTA takes the rows b, b + G, ... of the static assignment); 2 keeps
 * it on but makes every CTA of a forward run every queued segment (the path a
 * forward takes when its queue word is not its own). Process-wide, like the
 * override above; for comparing the assignments.
 */
rmsnorm_status rmsnorm_set_row_pool(int enabled);

/*
 * Shape of the row pool for later plans: percent of the rows in the per-CTA heads
 * (at >= 64 and at < 64 rows per CTA) and the longest and shortest segment
 * length; 0 keeps a default (85, 90, 16, 4). Process-wide, for tuning.
 */
rmsnorm_status rmsnorm_set_row_pool_shape(int head_pct, int head_pct_few, int len_max, int len_min);

/*
 * The row pool of M rows over G CTAs (head rows per CTA, segments in the queue;
 * head = 0: no pool), and rows [*first, *last) of its segment k. Host-only
 * arithmetic, no GPU needed.
 */
rmsnorm_status rmsnorm_row_pool_layout(int64_t M, int64_t G, int64_t* head, int64_t* nseg);
rmsnorm_status rmsnorm_row_pool_segment(int64_t M, int64_t G, int64_t k, int64_t* first, int64_t* last);

#ifdef __cplusplus
}
#endif
