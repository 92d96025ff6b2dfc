"""ctypes front end of the plain C RMSNorm oracle (``rmsnorm_oracle.c``).

TEST INFRASTRUCTURE: see the package docstring. Nothing here touches a GPU.

Arrays cross this boundary as numpy arrays in *storage* form: float32 data as
``np.float32``; float16 and bfloat16 data as their raw 16-bit patterns in
``np.uint16``. Golden results come back as ``np.float64``.

Every function mirrors one C function; the C file cites the passages each
formula follows. Parity status of each function is listed in ``PARITY``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPES = {"float32": 0, "float16": 1, "bfloat16": 2}
STORAGE = {"float32": np.float32, "float16": np.uint16, "bfloat16": np.uint16}

# Every oracle function is pinned by at least one test in tests/test_oracle_pins.py.
PARITY = {
    "fwd_golden": "pinned: printed worked examples, zero row, N=1 closed form, "
                  "scale invariance, library norm, 257-ones exercise",
    "bwd_golden": "pinned: printed dx example, finite differences, projection "
                  "identity, sum-not-mean table, zero row",
    "fwd_reference": "pinned: brute-force fp32 loop on tiny inputs, error bound vs golden",
    "bwd_reference": "pinned: brute-force fp32 loop on tiny inputs, error bound vs golden",
    "round/encode/decode": "pinned: numpy float16 and torch bfloat16 conversions, "
                           "hand-picked ties and overflow",
    "ln_fwd_golden": "pinned: hand-worked 4-element row, constant row, N=1, shift and "
                     "scale invariance, zero-mean rows match the RMSNorm golden",
    "ln_bwd_golden": "pinned: finite differences of the golden forward, per-row sums of dx "
                     "vanish, dbeta = column sums of dy, hand-worked 2-element row",
    "ln_fwd_reference": "pinned: brute-force fp32 loop on tiny inputs, error bound vs golden",
    "ln_bwd_reference": "pinned: brute-force fp32 loop on tiny inputs, error bound vs golden",
    "bwd_bwd_golden": "pinned: central finite differences of the (pinned) golden backward "
                      "contracted with ddx and ddgamma, for dy, x and gamma (plain and offset); "
                      "linearity in (ddx, ddgamma); zero cotangents give zero",
    "bwd_bwd_reference": "pinned: brute-force fp32 loop on tiny inputs, error bound vs golden",
    "dgamma_pairwise_reference": "pinned: brute-force fp32 pairwise loop on tiny inputs, "
                                 "log2(M) error bound vs golden",
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``rmsnorm_oracle.c`` with gcc (no FP contraction) if it is stale."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        F = ctypes.c_float
        sig = {
            "oracle_decode": [P, I, I64, P],
            "oracle_encode": [P, I64, I, P],
            "oracle_round": [P, I64, I, P],
            "oracle_fwd_golden": [P, P, I64, I64, D, I, I, P, P],
            "oracle_bwd_golden": [P, P, P, I64, I64, D, I, I, P, P],
            "oracle_fwd_reference": [P, P, I64, I64, F, I, I, P, P],
            "oracle_bwd_reference": [P, P, P, I64, I64, F, I, I, P, P],
            "oracle_ln_fwd_golden": [P, P, P, I64, I64, D, I, P, P, P],
            "oracle_ln_bwd_golden": [P, P, P, I64, I64, D, I, P, P, P],
            "oracle_ln_fwd_reference": [P, P, P, I64, I64, F, I, P, P, P],
            "oracle_ln_bwd_reference": [P, P, P, I64, I64, F, I, P, P, P],
            "oracle_bwd_bwd_golden": [P, P, P, P, P, I64, I64, D, I, I, P, P, P],
            "oracle_bwd_bwd_reference": [P, P, P, P, P, I64, I64, F, I, I, P, P, P],
            "oracle_dgamma_pairwise_reference": [P, P, P, I64, I64, F, I, I, P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(a, dtype, shape=None):
    a = np.ascontiguousarray(a)
    if a.dtype != STORAGE[dtype]:
        raise TypeError(f"expected storage {STORAGE[dtype]} for {dtype}, got {a.dtype}")
    if shape is not None and a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


# --------------------------------------------------------------------------- #
# number formats
# --------------------------------------------------------------------------- #
def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of an array stored as ``dtype``."""
    bits = _check(bits, dtype)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_decode(_ptr(bits), DTYPES[dtype], bits.size, _ptr(out))
    return out


def encode(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to nearest-even into ``dtype`` storage."""
    values = np.ascontiguousarray(values, np.float64)
    out = np.empty(values.shape, STORAGE[dtype])
    _load().oracle_encode(_ptr(values), values.size, DTYPES[dtype], _ptr(out))
    return out


def round_to(values: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> dtype (nearest-even) -> fp64, i.e. ``golden.to(dtype).to(fp64)``."""
    values = np.ascontiguousarray(values, np.float64)
    out = np.empty(values.shape, np.float64)
    _load().oracle_round(_ptr(values), values.size, DTYPES[dtype], _ptr(out))
    return out


# --------------------------------------------------------------------------- #
# golden (fp64)
# --------------------------------------------------------------------------- #
def fwd_golden(x, gamma, dtype, eps=1e-6, offset=False, want_y=True):
    """Returns ``(y fp64 [M,N] or None, rstd fp64 [M])``."""
    x = _check(x, dtype)
    M, N = x.shape
    gamma = _check(gamma, dtype, (N,))
    y = np.empty((M, N), np.float64) if want_y else None
    rstd = np.empty(M, np.float64)
    _load().oracle_fwd_golden(_ptr(x), _ptr(gamma), M, N, float(eps), DTYPES[dtype],
                              int(bool(offset)), _ptr(y), _ptr(rstd))
    return y, rstd


def bwd_golden(dy, x, gamma, dtype, eps=1e-6, offset=False, want_dx=True):
    """Returns ``(dx fp64 [M,N] or None, dgamma fp64 [N])``."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    dx = np.empty((M, N), np.float64) if want_dx else None
    dg = np.empty(N, np.float64)
    _load().oracle_bwd_golden(_ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                              DTYPES[dtype], int(bool(offset)), _ptr(dx), _ptr(dg))
    return dx, dg


# --------------------------------------------------------------------------- #
# reference (I/O dtype, fp32 intermediates)
# --------------------------------------------------------------------------- #
def fwd_reference(x, gamma, dtype, eps=1e-6, offset=False):
    """Returns ``(y [M,N] in dtype storage, rstd float32 [M])``."""
    x = _check(x, dtype)
    M, N = x.shape
    gamma = _check(gamma, dtype, (N,))
    y = np.empty((M, N), STORAGE[dtype])
    rstd = np.empty(M, np.float32)
    _load().oracle_fwd_reference(_ptr(x), _ptr(gamma), M, N, float(eps), DTYPES[dtype],
                                 int(bool(offset)), _ptr(y), _ptr(rstd))
    return y, rstd


def bwd_reference(dy, x, gamma, dtype, eps=1e-6, offset=False, want_dx=True):
    """Returns ``(dx [M,N] in dtype storage or None, dgamma [N] in dtype storage)``."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    dx = np.empty((M, N), STORAGE[dtype]) if want_dx else None
    dg = np.empty(N, STORAGE[dtype])
    _load().oracle_bwd_reference(_ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                                 DTYPES[dtype], int(bool(offset)), _ptr(dx), _ptr(dg))
    return dx, dg


# --------------------------------------------------------------------------- #
# LayerNorm (golden fp64; reference in the I/O dtype with fp32 intermediates)
# --------------------------------------------------------------------------- #
def ln_fwd_golden(x, gamma, beta, dtype, eps=1e-5, want_y=True):
    """Returns ``(y fp64 [M,N] or None, mean fp64 [M], rstd fp64 [M])``."""
    x = _check(x, dtype)
    M, N = x.shape
    gamma = _check(gamma, dtype, (N,))
    beta = _check(beta, dtype, (N,))
    y = np.empty((M, N), np.float64) if want_y else None
    mean = np.empty(M, np.float64)
    rstd = np.empty(M, np.float64)
    _load().oracle_ln_fwd_golden(_ptr(x), _ptr(gamma), _ptr(beta), M, N, float(eps),
                                 DTYPES[dtype], _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def ln_bwd_golden(dy, x, gamma, dtype, eps=1e-5, want_dx=True):
    """Returns ``(dx fp64 [M,N] or None, dgamma fp64 [N], dbeta fp64 [N])``."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    dx = np.empty((M, N), np.float64) if want_dx else None
    dg = np.empty(N, np.float64)
    db = np.empty(N, np.float64)
    _load().oracle_ln_bwd_golden(_ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                                 DTYPES[dtype], _ptr(dx), _ptr(dg), _ptr(db))
    return dx, dg, db


def ln_fwd_reference(x, gamma, beta, dtype, eps=1e-5):
    """Returns ``(y [M,N] in dtype storage, mean float32 [M], rstd float32 [M])``."""
    x = _check(x, dtype)
    M, N = x.shape
    gamma = _check(gamma, dtype, (N,))
    beta = _check(beta, dtype, (N,))
    y = np.empty((M, N), STORAGE[dtype])
    mean = np.empty(M, np.float32)
    rstd = np.empty(M, np.float32)
    _load().oracle_ln_fwd_reference(_ptr(x), _ptr(gamma), _ptr(beta), M, N, float(eps),
                                    DTYPES[dtype], _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def ln_bwd_reference(dy, x, gamma, dtype, eps=1e-5, want_dx=True):
    """Returns ``(dx or None, dgamma, dbeta)`` in dtype storage."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    dx = np.empty((M, N), STORAGE[dtype]) if want_dx else None
    dg = np.empty(N, STORAGE[dtype])
    db = np.empty(N, STORAGE[dtype])
    _load().oracle_ln_bwd_reference(_ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                                    DTYPES[dtype], _ptr(dx), _ptr(dg), _ptr(db))
    return dx, dg, db


# --------------------------------------------------------------------------- #
# RMSNorm double backward
# --------------------------------------------------------------------------- #
def bwd_bwd_golden(ddx, ddg, dy, x, gamma, dtype, eps=1e-6, offset=False):
    """Gradients of sum(ddx*dx) + sum(ddg*dgamma) for dy, x and gamma, fp64.
    ddg may be None (zero). Returns ``(d_dy [M,N], d_x [M,N], d_gamma [N])``."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    ddx = _check(ddx, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    if ddg is not None:
        ddg = _check(ddg, dtype, (N,))
    d_dy = np.empty((M, N), np.float64)
    d_x = np.empty((M, N), np.float64)
    d_g = np.empty(N, np.float64)
    _load().oracle_bwd_bwd_golden(_ptr(ddx), _ptr(ddg), _ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                                  DTYPES[dtype], int(bool(offset)), _ptr(d_dy), _ptr(d_x), _ptr(d_g))
    return d_dy, d_x, d_g


def bwd_bwd_reference(ddx, ddg, dy, x, gamma, dtype, eps=1e-6, offset=False):
    """Same in dtype storage with fp32 intermediates."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    ddx = _check(ddx, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    if ddg is not None:
        ddg = _check(ddg, dtype, (N,))
    d_dy = np.empty((M, N), STORAGE[dtype])
    d_x = np.empty((M, N), STORAGE[dtype])
    d_g = np.empty(N, STORAGE[dtype])
    _load().oracle_bwd_bwd_reference(_ptr(ddx), _ptr(ddg), _ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps),
                                     DTYPES[dtype], int(bool(offset)), _ptr(d_dy), _ptr(d_x), _ptr(d_g))
    return d_dy, d_x, d_g


def dgamma_pairwise_reference(dy, x, gamma, dtype, eps=1e-6, offset=False):
    """dgamma [N] in dtype storage: fp32 terms summed over rows by a pairwise tree."""
    x = _check(x, dtype)
    M, N = x.shape
    dy = _check(dy, dtype, (M, N))
    gamma = _check(gamma, dtype, (N,))
    dg = np.empty(N, STORAGE[dtype])
    _load().oracle_dgamma_pairwise_reference(_ptr(dy), _ptr(x), _ptr(gamma), M, N, float(eps), DTYPES[dtype],
                                             int(bool(offset)), _ptr(dg))
    return dg
