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

#ifdef __cplusplus
}
#endif
