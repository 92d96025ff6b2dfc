"""Seeded synthetic inputs and the workload table.

This module is shared by the GPU tests, the oracle tests and the benchmark. It
holds none of the RMSNorm or LayerNorm arithmetic: it only draws random numbers and stores
them in the I/O dtype (round-to-nearest-even, done by numpy for float16 and by
torch for bfloat16). It imports neither the GPU library nor the oracle.

Recipe (every tensor gets its own random stream):
  * stream key = SeedSequence([seed, tag]) with tag 0 for x, 1 for gamma/w,
    2 for dy, 3 and 4 for the extra draws of the adversarial rows; bit
    generator PCG64; samples drawn in float32.
  * x ~ x_scale * N(0,1); gamma = 1 + 0.1 * N(0,1) (offset variant: w = 0.05 * N(0,1));
    dy ~ dy_scale * N(0,1).
  * adversarial rows: row i has class i mod 5 --
      0 all zero; 1 constant 1e4; 2 1e-20 * N(0,1);
      3 N(0,1) with one outlier 6e4 at column (i * 7919) mod N; 4 uniform[-1, 1).
  * LayerNorm inputs: x = row_shift * s_i + x_scale * N(0,1), with one shift
    s_i ~ N(0,1) per row (tag 5) so that rows have non-zero means;
    gamma = 1 + 0.1 * N(0,1); beta = 0.1 * N(0,1) (tag 6); dy as above.

Storage form (what the oracle and the GPU tests exchange): float32 data as
np.float32, float16/bfloat16 as raw 16-bit patterns in np.uint16.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TAG_X, TAG_GAMMA, TAG_DY, TAG_ADV_U, TAG_ADV_Z, TAG_SHIFT, TAG_BETA = 0, 1, 2, 3, 4, 5, 6
ELEM_BYTES = {"float32": 4, "float16": 2, "bfloat16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    dtype: str
    offset: bool = False
    x_scale: float = 1.0
    dy_scale: float = 1.0
    adversarial: bool = False
    seed: int = 0
    eps: float = 1e-6
    op: str = "rmsnorm"          # or "layernorm"
    row_shift: float = 0.0       # LayerNorm inputs: spread of the per-row means

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    def fwd_bytes(self) -> int:
        """Algorithmic HBM bytes of one forward. RMSNorm: read x and gamma, write y
        and rstd. LayerNorm: also read beta and write mean."""
        s = self.elem_bytes
        if self.op == "layernorm":
            return 2 * self.M * self.N * s + 2 * self.N * s + 8 * self.M
        return 2 * self.M * self.N * s + self.N * s + 4 * self.M

    def bwd_bytes(self) -> int:
        """Algorithmic HBM bytes of one backward: read x, dy, write dx, read gamma,
        write dgamma, read rstd (the dgamma partials are overhead, not counted).
        LayerNorm: also read mean and write dbeta."""
        s = self.elem_bytes
        if self.op == "layernorm":
            return 3 * self.M * self.N * s + 3 * self.N * s + 8 * self.M
        return 3 * self.M * self.N * s + 2 * self.N * s + 4 * self.M


# The workloads the library is measured and gated on.
WORKLOADS = {w.name: w for w in [
    Workload("fp32_64x256", 64, 256, "float32"),
    Workload("bf16_4096x4096", 4096, 4096, "bfloat16"),
    Workload("bf16_65536x4096", 65536, 4096, "bfloat16", x_scale=3.0, dy_scale=1e-2),
    Workload("fp16_offset_16384x8192", 16384, 8192, "float16", offset=True),
    Workload("fp16_offset_16384x16384", 16384, 16384, "float16", offset=True),
    Workload("fp32_offset_16384x8192", 16384, 8192, "float32", offset=True),
    Workload("fp32_offset_16384x16384", 16384, 16384, "float32", offset=True),
    Workload("bf16_adversarial_8192x5120", 8192, 5120, "bfloat16", adversarial=True),
    Workload("bf16_adversarial_8192x4099", 8192, 4099, "bfloat16", adversarial=True),
    Workload("ln_bf16_65536x4096", 65536, 4096, "bfloat16", eps=1e-5, op="layernorm", row_shift=2.0),
    Workload("ln_fp32_16384x16384", 16384, 16384, "float32", eps=1e-5, op="layernorm", row_shift=2.0),
    Workload("ln_bf16_16384x4099", 16384, 4099, "bfloat16", eps=1e-5, op="layernorm", row_shift=2.0),
    # narrow rows (a row per group of lanes)
    Workload("bf16_1048576x128", 1 << 20, 128, "bfloat16"),
    Workload("ln_bf16_524288x256", 524288, 256, "bfloat16", eps=1e-5, op="layernorm", row_shift=2.0),
]}

HEADLINE = "bf16_65536x4096"


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


def to_storage(values: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage form of ``dtype`` (nearest-even)."""
    values = np.ascontiguousarray(values, np.float32)
    if dtype == "float32":
        return values
    if dtype == "float16":
        return values.astype(np.float16).view(np.uint16)
    if dtype == "bfloat16":
        import torch
        t = torch.from_numpy(values).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def normal(seed: int, tag: int, shape, scale: float = 1.0) -> np.ndarray:
    z = _rng(seed, tag).standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        z *= np.float32(scale)
    return z


def adversarial_rows(M: int, N: int, seed: int) -> np.ndarray:
    """float32 matrix whose row i follows class i mod 5 (see module docstring)."""
    z = normal(seed, TAG_X, (M, N))
    cls = np.arange(M) % 5
    out = np.empty((M, N), np.float32)
    out[cls == 0] = 0.0
    out[cls == 1] = 1e4
    tiny = normal(seed, TAG_ADV_Z, (M, N))
    out[cls == 2] = tiny[cls == 2] * np.float32(1e-20)
    rows3 = np.nonzero(cls == 3)[0]
    out[rows3] = z[rows3]
    out[rows3, (rows3 * 7919) % N] = 6e4
    uni = _rng(seed, TAG_ADV_U).uniform(-1.0, 1.0, (M, N)).astype(np.float32)
    out[cls == 4] = uni[cls == 4]
    return out


def make_inputs(M: int, N: int, dtype: str, *, seed: int = 0, offset: bool = False,
                x_scale: float = 1.0, dy_scale: float = 1.0, adversarial: bool = False):
    """Returns storage-form ``x [M,N]``, ``gamma [N]`` (w for the offset variant), ``dy [M,N]``."""
    if adversarial:
        xf = adversarial_rows(M, N, seed)
    else:
        xf = normal(seed, TAG_X, (M, N), x_scale)
    if offset:
        gf = normal(seed, TAG_GAMMA, (N,), 0.05)
    else:
        gf = np.float32(1.0) + normal(seed, TAG_GAMMA, (N,), 0.1)
    dyf = normal(seed, TAG_DY, (M, N), dy_scale)
    return to_storage(xf, dtype), to_storage(gf, dtype), to_storage(dyf, dtype)


def make_ln_inputs(M: int, N: int, dtype: str, *, seed: int = 0, x_scale: float = 1.0,
                   row_shift: float = 2.0, dy_scale: float = 1.0):
    """LayerNorm inputs: storage-form ``x [M,N]``, ``gamma [N]``, ``beta [N]``, ``dy [M,N]``."""
    xf = normal(seed, TAG_X, (M, N), x_scale)
    if row_shift:
        xf += normal(seed, TAG_SHIFT, (M, 1), row_shift)
    gf = np.float32(1.0) + normal(seed, TAG_GAMMA, (N,), 0.1)
    bf = normal(seed, TAG_BETA, (N,), 0.1)
    dyf = normal(seed, TAG_DY, (M, N), dy_scale)
    return to_storage(xf, dtype), to_storage(gf, dtype), to_storage(bf, dtype), to_storage(dyf, dtype)


def workload_inputs(w: Workload):
    if w.op == "layernorm":
        return make_ln_inputs(w.M, w.N, w.dtype, seed=w.seed, x_scale=w.x_scale,
                              row_shift=w.row_shift, dy_scale=w.dy_scale)
    return make_inputs(w.M, w.N, w.dtype, seed=w.seed, offset=w.offset,
                       x_scale=w.x_scale, dy_scale=w.dy_scale, adversarial=w.adversarial)
