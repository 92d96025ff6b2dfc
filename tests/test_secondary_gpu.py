"""The pages' secondary numerical reports, on the GPU through the C ABI.

1. The closeness check of the page "Check an AI model calculation before
   accelerating it" (section "Measurements before results", "Three distinct
   numerical comparisons"): 72 cases each for the forward output, dx and
   dgamma, each compared element by element with the same-dtype reference at
   the tolerances the page declares (FP32 atol 1e-5 / rtol 1e-4, FP16
   atol = rtol = 3e-3; the page declares none for bfloat16, which the main gate
   covers). The 72 cases: 18 shapes x {float32, float16} x {plain, offset}.
   Reported beside the golden/reference/target gate, not instead of it.
2. The growth study of dgamma's error over the reduction length M (page
   "torchtitan kernel numerics verification", the conditioning check's
   alternative analysis): M = 2^10 .. 2^16, three seeds, float32 I/O so that
   the accumulation error is not hidden by an output rounding; the kernel's
   growth is judged against the sequential fp32 reference's.
"""
import numpy as np
import pytest

from oracle import gate, growth
from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util

pytestmark = pytest.mark.gpu

# shapes: the torchtitan page's tile-boundary table (flattened), the checking
# page's benchmark shape 128 x 257, the smallest legal shapes and one row of each
# kernel path (lanes, ring, ragged, row-vector, wide rows)
SHAPES = [(1, 1), (1, 2), (64, 1), (3, 255), (3, 256), (3, 257), (48, 256), (8, 4095), (8, 4096),
          (8, 4097), (8, 5120), (128, 257), (17, 1000), (33, 768), (9, 2048), (5, 8192), (3, 16384),
          (1000, 128)]
CASES = [(shape, dtype, offset) for dtype in ("float32", "float16") for offset in (False, True)
         for shape in SHAPES]
assert len(CASES) == 72


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fwd_bwd_gb300 import binding
    binding.rmsnorm_device_error(clear=True)
    yield
    assert binding.rmsnorm_device_error(clear=True) == 0


def test_closeness_check_72_cases_each():
    rows = ["| case | y failing / worst excess | dx failing / worst excess | dgamma failing / worst excess |",
            "|---|---|---|---|"]
    failures = []
    for i, ((M, N), dtype, offset) in enumerate(CASES):
        x, g, dy = inputs.make_inputs(M, N, dtype, seed=100 + i, offset=offset)
        y, _, dx, dg = gpu_util.run(x, g, dy, dtype, offset=offset)
        yr, _ = orc.fwd_reference(x, g, dtype, offset=offset)
        dxr, dgr = orc.bwd_reference(dy, x, g, dtype, offset=offset)
        res = [gate.allclose(name, orc.decode(t, dtype), orc.decode(r, dtype), dtype)
               for name, t, r in (("y", y, yr), ("dx", dx, dxr), ("dgamma", dg, dgr))]
        rows.append(f"| {dtype} {M}x{N}{' offset' if offset else ''} | "
                    + " | ".join(f"{r.failing}/{r.elements} {r.worst_excess:.2e}" for r in res) + " |")
        failures += [f"{dtype} {M}x{N} offset={offset} {r.tensor}: {r.failing} elements"
                     for r in res if not r.passed]
    print("\n" + "\n".join(rows))
    print(f"closeness check: {3 * len(CASES) - len(failures)} of {3 * len(CASES)} comparisons pass")
    assert not failures, failures


def test_dgamma_error_growth_over_rows():
    N = 1024
    target, seq, pw = growth.Series("kernel"), growth.Series("sequential fp32"), growth.Series("pairwise fp32")
    conditions = {}
    for k in range(10, 17):
        M = 1 << k
        conds = []
        for seed in range(3):
            x, g, dy = inputs.make_inputs(M, N, "float32", seed=seed)
            _, _, _, dg = gpu_util.run(x, g, dy, "float32")
            _, gold = orc.bwd_golden(dy, x, g, "float32", want_dx=False)
            _, ref = orc.bwd_reference(dy, x, g, "float32", want_dx=False)
            target.add(M, seed, orc.decode(dg, "float32"), gold)
            seq.add(M, seed, orc.decode(ref, "float32"), gold)
            pw.add(M, seed, orc.decode(orc.dgamma_pairwise_reference(dy, x, g, "float32"), "float32"), gold)
            _, r = orc.fwd_golden(x, g, "float32", want_y=False)
            xd, dyd = orc.decode(x[:, :64], "float32"), orc.decode(dy[:, :64], "float32")
            conds += [gate.condition_number(dyd[:, j] * xd[:, j] * r) for j in range(64)]
        conditions[M] = float(np.median(conds))
    v = growth.judge(target, seq)
    print("\n" + growth.report("dgamma error growth, float32, N = 1024", [target, seq, pw], conditions, v))
    assert v.verdict == "PASS WITH LIMITATIONS", v.notes
