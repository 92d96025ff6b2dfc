"""Cases run against the debug build of the library (librmsnorm_debug.so, built
with -DRMSNORM_DEBUG): every TMA read of a row kernel is first checked against
the extent of the tensor it reads, and a read outside it sets bit 1 of the
device error word. Run as ``RMSNORM_LIBRARY=<debug .so> python -m
tests.debug_build_cases``: each case is gated against the oracle and the error
word must stay 0. Covers every path that reads with TMA copies: the aligned ring
(one CTA and clusters), the row pool's kernels, the ragged ring at shifted pointers
and odd pitches, LayerNorm and the double backward, plus the lane-group and
row-vector paths.
"""
import sys


from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util


def main() -> int:
    import torch
    assert torch.cuda.is_available()
    assert B.LIB_PATH.endswith("librmsnorm_debug.so"), B.LIB_PATH
    B.rmsnorm_device_error(clear=True)
    results = []
    # RMSNorm: aligned ring, clusters, ragged (dense, shifted), row-vector, lanes
    # (and the row pool's forward and backward, 10001 rows: heads, then queued
    # segments, the last one short)
    for M, N, dt, off, mis in ((67, 4096, "bfloat16", False, False), (9, 16384, "float32", True, False),
                               (37, 4099, "bfloat16", False, False), (29, 4099, "float32", True, False),
                               (33, 4096, "bfloat16", False, True), (41, 2051, "float16", False, True),
                               (13, 9999, "bfloat16", False, False), (257, 256, "bfloat16", False, False),
                               (10001, 4096, "bfloat16", True, False)):
        x, g, dy = inputs.make_inputs(M, N, dt, seed=M + N, offset=off)
        y, r, dx, dg = gpu_util.run(x, g, dy, dt, offset=off, misalign={"x", "dy"} if mis else False)
        results += check.gate_outputs(x, g, dy, dt, off, 1e-6, y=y, rstd=r, dx=dx, dgamma=dg)
    # strided rows at odd pitches (ragged ring with a pitch that is not a 16-byte multiple)
    M, N, ld = 31, 4099, 4105
    x, g, dy = inputs.make_inputs(M, N, "bfloat16", seed=7)
    xb = torch.zeros((M, ld), dtype=torch.bfloat16, device="cuda")
    dyb = torch.zeros((M, ld), dtype=torch.bfloat16, device="cuda")
    xb[:, :N] = B.to_device(x.reshape(-1), "bfloat16").view(M, N)
    dyb[:, :N] = B.to_device(dy.reshape(-1), "bfloat16").view(M, N)
    gt = B.to_device(g, "bfloat16")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(y)
    dg = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    assert B.rmsnorm_fwd_strided(xb, ld, gt, y, N, r, M, N, 1e-6, "bfloat16", 0) == 0
    wsz = B.rmsnorm_bwd_workspace_size(M, N, "bfloat16")
    ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_bwd_strided(dyb, ld, xb, ld, gt, r, dx, N, dg, M, N, "bfloat16", 0, ws, wsz) == 0
    torch.cuda.synchronize()
    results += check.gate_outputs(x, g, dy, "bfloat16", False, 1e-6, y=B.to_numpy(y, "bfloat16").reshape(M, N),
                                  rstd=B.to_numpy(r, "float32"), dx=B.to_numpy(dx, "bfloat16").reshape(M, N),
                                  dgamma=B.to_numpy(dg, "bfloat16"))
    # LayerNorm: aligned ring, ragged ring
    for M, N in ((64, 4096), (33, 4099)):
        x, g, b, dy = inputs.make_ln_inputs(M, N, "bfloat16", seed=M)
        y, mean, rstd, dx, dgm, dbt = gpu_util.ln_run(x, g, b, dy, "bfloat16")
        results += check.gate_ln_outputs(x, g, b, dy, "bfloat16", 1e-5, y=y, mean=mean, rstd=rstd, dx=dx,
                                         dgamma=dgm, dbeta=dbt)
    # double backward: aligned ring, ragged ring
    for M, N in ((64, 2048), (35, 4099)):
        x, g, dy = inputs.make_inputs(M, N, "bfloat16", seed=N)
        ddx = inputs.to_storage(inputs.normal(0, 3, (M, N)), "bfloat16")
        ddg = inputs.to_storage(inputs.normal(0, 4, (N,)), "bfloat16")
        d_dy, d_x, d_g = gpu_util.dbwd_run(ddx, ddg, dy, x, g, "bfloat16")
        results += check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, "bfloat16", False, 1e-6, d_dy=d_dy, d_x=d_x,
                                              d_gamma=d_g)
    word = B.rmsnorm_device_error(clear=True)
    verdict = gate.overall(results)
    print(f"debug build: {len(results)} gated tensors, overall {verdict}, device error word {word}")
    return 0 if (word == 0 and verdict == "PASS" and results) else 1


if __name__ == "__main__":
    sys.exit(main())
