"""Python front end of ``librmsnorm.so`` (the C ABI in ``include/rmsnorm.h``,
``include/layernorm.h`` and ``include/rmsnorm_double_backward.h``).

The functions named like the C entry points take the same arguments in the same
order and only marshal them: a pointer argument may be a torch tensor (its
``data_ptr()``), an int address or ``None``; ``dtype`` may be an
``rmsnorm_dtype`` code, a dtype name or a ``torch.dtype``; ``stream`` may be a
``torch.cuda.Stream``, a raw handle or ``None`` (torch's current stream). They
return the C status code. All computation happens in the library's CUDA
kernels; there is no other code path. If the library is missing, every call
raises ``RuntimeError``.

``forward``/``backward`` are conveniences for torch tensors that allocate the
outputs (and the backward workspace) with torch and raise ``RMSNormError`` on a
non-OK status.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# RMSNORM_LIBRARY may name another build of this library (the debug build,
# librmsnorm_debug.so, whose kernels check their reads); default: the release build.
LIB_PATH = os.environ.get("RMSNORM_LIBRARY") or os.path.join(HERE, "librmsnorm.so")
INCLUDE_DIR = os.path.join(os.path.dirname(HERE), "include")
HEADER_PATH = os.path.join(INCLUDE_DIR, "rmsnorm.h")

RMSNORM_F32, RMSNORM_F16, RMSNORM_BF16 = 0, 1, 2
DTYPE_CODES = {"float32": RMSNORM_F32, "float16": RMSNORM_F16, "bfloat16": RMSNORM_BF16}
ELEM_BYTES = {RMSNORM_F32: 4, RMSNORM_F16: 2, RMSNORM_BF16: 2}
STATUS_NAMES = {
    0: "RMSNORM_OK", 1: "RMSNORM_ERR_NULL", 2: "RMSNORM_ERR_SHAPE", 3: "RMSNORM_ERR_DTYPE",
    4: "RMSNORM_ERR_EPS", 5: "RMSNORM_ERR_ALIGN", 6: "RMSNORM_ERR_WORKSPACE",
    7: "RMSNORM_ERR_UNSUPPORTED", 8: "RMSNORM_ERR_CUDA", 9: "RMSNORM_ERR_ARG",
}
RMSNORM_OK = 0

_lock = threading.Lock()
_lib = None


class RMSNormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({rmsnorm_status_string(status)})")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I, F, SZ, U32P = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                  ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32))
        sigs = {
            "rmsnorm_fwd": (I, [P, P, P, P, I64, I64, F, I, I, P]),
            "rmsnorm_bwd_workspace_size": (SZ, [I64, I64, I]),
            "rmsnorm_bwd": (I, [P, P, P, P, P, P, I64, I64, I, I, P, SZ, P]),
            "rmsnorm_status_string": (ctypes.c_char_p, [I]),
            "rmsnorm_device_error": (I, [U32P, I]),
            "rmsnorm_describe_plan": (I, [I, I64, I64, I, I, ctypes.c_char_p, SZ]),
            "rmsnorm_set_launch_override": (I, [I, I, I, I, I]),
            "rmsnorm_set_row_pool": (I, [I]),
            "rmsnorm_set_row_pool_shape": (I, [I, I, I, I]),
            "rmsnorm_row_pool_layout": (I, [I64, I64, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
            "rmsnorm_row_pool_segment": (I, [I64, I64, I64, ctypes.POINTER(ctypes.c_int64),
                                             ctypes.POINTER(ctypes.c_int64)]),
            "rmsnorm_bwd_static_scratch": (I, [P, P, P, P, P, P, I64, I64, I, I, P]),
            "rmsnorm_selftest_wait_timeout": (I, [ctypes.c_uint32, P]),
            "rmsnorm_fwd_strided": (I, [P, I64, P, P, I64, P, I64, I64, F, I, I, P]),
            "rmsnorm_bwd_strided": (I, [P, I64, P, I64, P, P, P, I64, P, I64, I64, I, I, P, SZ, P]),
            "layernorm_fwd": (I, [P, I64, P, P, P, I64, P, P, I64, I64, F, I, P]),
            "layernorm_bwd_workspace_size": (SZ, [I64, I64, I]),
            "layernorm_bwd": (I, [P, I64, P, I64, P, P, P, P, I64, P, P, I64, I64, I, P, SZ, P]),
            "rmsnorm_bwd_bwd_workspace_size": (SZ, [I64, I64, I]),
            "rmsnorm_bwd_bwd": (I, [P, I64, P, P, I64, P, I64, P, P, P, I64, P, I64, P, I64, I64, I, I, P, SZ,
                                    P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def header_functions() -> list:
    """Names of the functions declared in include/*.h."""
    names = set()
    for fn in sorted(os.listdir(INCLUDE_DIR)):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(INCLUDE_DIR, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b((?:rmsnorm|layernorm)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def _addr(p):
    if p is None:
        return None
    if isinstance(p, int):
        return p
    if hasattr(p, "data_ptr"):
        return p.data_ptr()
    raise TypeError(f"cannot take the address of {type(p)}")


def _dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    if isinstance(dt, str):
        return DTYPE_CODES[dt]
    name = str(dt).replace("torch.", "")
    return DTYPE_CODES[name]


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# --------------------------------------------------------------------------- #
# the C entry points
# --------------------------------------------------------------------------- #
def rmsnorm_fwd(x, gamma, y, rstd, M, N, eps, dtype, offset, stream=None) -> int:
    return _load().rmsnorm_fwd(_addr(x), _addr(gamma), _addr(y), _addr(rstd), int(M), int(N),
                               float(eps), _dtype_code(dtype), int(offset), _stream(stream))


def rmsnorm_fwd_strided(x, ldx, gamma, y, ldy, rstd, M, N, eps, dtype, offset, stream=None) -> int:
    return _load().rmsnorm_fwd_strided(_addr(x), int(ldx), _addr(gamma), _addr(y), int(ldy), _addr(rstd),
                                       int(M), int(N), float(eps), _dtype_code(dtype), int(offset),
                                       _stream(stream))


def rmsnorm_bwd_strided(dy, lddy, x, ldx, gamma, rstd, dx, lddx, dgamma, M, N, dtype, offset, workspace,
                        workspace_bytes, stream=None) -> int:
    return _load().rmsnorm_bwd_strided(_addr(dy), int(lddy), _addr(x), int(ldx), _addr(gamma), _addr(rstd),
                                       _addr(dx), int(lddx), _addr(dgamma), int(M), int(N),
                                       _dtype_code(dtype), int(offset), _addr(workspace),
                                       int(workspace_bytes), _stream(stream))


def rmsnorm_bwd_workspace_size(M, N, dtype) -> int:
    return int(_load().rmsnorm_bwd_workspace_size(int(M), int(N), _dtype_code(dtype)))


def rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, offset, workspace, workspace_bytes,
                stream=None) -> int:
    return _load().rmsnorm_bwd(_addr(dy), _addr(x), _addr(gamma), _addr(rstd), _addr(dx),
                               _addr(dgamma), int(M), int(N), _dtype_code(dtype), int(offset),
                               _addr(workspace), int(workspace_bytes), _stream(stream))


def rmsnorm_bwd_static_scratch(dy, x, gamma, rstd, dx, dgamma, M, N, dtype, offset,
                               stream=None) -> int:
    """rmsnorm_bwd without a workspace argument: for callers that cannot allocate
    device memory (the partial sums live in a fixed array inside the library)."""
    return _load().rmsnorm_bwd_static_scratch(_addr(dy), _addr(x), _addr(gamma), _addr(rstd),
                                              _addr(dx), _addr(dgamma), int(M), int(N),
                                              _dtype_code(dtype), int(offset), _stream(stream))


def layernorm_fwd(x, ldx, gamma, beta, y, ldy, mean, rstd, M, N, eps, dtype, stream=None) -> int:
    return _load().layernorm_fwd(_addr(x), int(ldx), _addr(gamma), _addr(beta), _addr(y), int(ldy),
                                 _addr(mean), _addr(rstd), int(M), int(N), float(eps), _dtype_code(dtype),
                                 _stream(stream))


def layernorm_bwd_workspace_size(M, N, dtype) -> int:
    return int(_load().layernorm_bwd_workspace_size(int(M), int(N), _dtype_code(dtype)))


def layernorm_bwd(dy, lddy, x, ldx, gamma, mean, rstd, dx, lddx, dgamma, dbeta, M, N, dtype, workspace,
                  workspace_bytes, stream=None) -> int:
    return _load().layernorm_bwd(_addr(dy), int(lddy), _addr(x), int(ldx), _addr(gamma), _addr(mean),
                                 _addr(rstd), _addr(dx), int(lddx), _addr(dgamma), _addr(dbeta), int(M),
                                 int(N), _dtype_code(dtype), _addr(workspace), int(workspace_bytes),
                                 _stream(stream))


def rmsnorm_bwd_bwd_workspace_size(M, N, dtype) -> int:
    return int(_load().rmsnorm_bwd_bwd_workspace_size(int(M), int(N), _dtype_code(dtype)))


def rmsnorm_bwd_bwd(ddx, ldddx, ddgamma, dy, lddy, x, ldx, gamma, rstd, d_dy, ldd_dy, d_x, ldd_x, d_gamma, M, N,
                    dtype, offset, workspace, workspace_bytes, stream=None) -> int:
    return _load().rmsnorm_bwd_bwd(_addr(ddx), int(ldddx), _addr(ddgamma), _addr(dy), int(lddy), _addr(x),
                                   int(ldx), _addr(gamma), _addr(rstd), _addr(d_dy), int(ldd_dy), _addr(d_x),
                                   int(ldd_x), _addr(d_gamma), int(M), int(N), _dtype_code(dtype), int(offset),
                                   _addr(workspace), int(workspace_bytes), _stream(stream))


def rmsnorm_status_string(status: int) -> str:
    return _load().rmsnorm_status_string(int(status)).decode()


def rmsnorm_device_error(clear: bool = False) -> int:
    flags = ctypes.c_uint32(0)
    st = _load().rmsnorm_device_error(ctypes.byref(flags), int(bool(clear)))
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_device_error")
    return int(flags.value)


def rmsnorm_selftest_wait_timeout(polls, stream=None) -> int:
    return _load().rmsnorm_selftest_wait_timeout(int(polls), _stream(stream))


def rmsnorm_describe_plan(pass_, M, N, dtype, aligned16=True) -> str:
    """aligned16: True/1 aligned, False/0 shared 16-byte offset, 2 mixed offsets."""
    buf = ctypes.create_string_buffer(256)
    st = _load().rmsnorm_describe_plan(int(pass_), int(M), int(N), _dtype_code(dtype),
                                       int(aligned16), buf, 256)
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_describe_plan")
    return buf.value.decode()


def rmsnorm_set_launch_override(pass_, threads=0, vpt=0, stages=0, blocks_per_sm=0) -> int:
    return _load().rmsnorm_set_launch_override(int(pass_), int(threads), int(vpt), int(stages),
                                               int(blocks_per_sm))


def rmsnorm_set_row_pool(enabled) -> int:
    """0/False: static rows; 1/True: the row pool; 2: pool with the forward's queue bypassed."""
    return _load().rmsnorm_set_row_pool(int(enabled))


def rmsnorm_set_row_pool_shape(head_pct=0, head_pct_few=0, len_max=0, len_min=0) -> int:
    return _load().rmsnorm_set_row_pool_shape(int(head_pct), int(head_pct_few), int(len_max), int(len_min))


def rmsnorm_row_pool_layout(M: int, G: int):
    """(head rows per CTA, segments in the queue) of the backward's row pool."""
    head, nseg = ctypes.c_int64(), ctypes.c_int64()
    st = _load().rmsnorm_row_pool_layout(int(M), int(G), ctypes.byref(head), ctypes.byref(nseg))
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_row_pool_layout")
    return head.value, nseg.value


def rmsnorm_row_pool_segment(M: int, G: int, k: int):
    """Rows [first, last) of segment k of the backward's row pool."""
    first, last = ctypes.c_int64(), ctypes.c_int64()
    st = _load().rmsnorm_row_pool_segment(int(M), int(G), int(k), ctypes.byref(first), ctypes.byref(last))
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_row_pool_segment")
    return first.value, last.value


# --------------------------------------------------------------------------- #
# torch conveniences
# --------------------------------------------------------------------------- #
def forward(x, gamma, eps: float = 1e-6, offset: bool = False, stream=None):
    """y, rstd = RMSNorm(x) for a contiguous CUDA tensor x[..., N]."""
    import torch
    if not (x.is_cuda and gamma.is_cuda and x.is_contiguous() and gamma.is_contiguous()):
        raise ValueError("x and gamma must be contiguous CUDA tensors")
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    y = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = rmsnorm_fwd(x, gamma, y, rstd, M, N, eps, x.dtype, int(offset), stream)
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_fwd")
    return y, rstd


def backward(dy, x, gamma, rstd, offset: bool = False, stream=None, workspace=None):
    """dx, dgamma for a contiguous CUDA tensor x[..., N] and the forward's rstd."""
    import torch
    for t in (dy, x, gamma, rstd):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    need = rmsnorm_bwd_workspace_size(M, N, x.dtype)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    dx = torch.empty_like(x)
    dgamma = torch.empty_like(gamma)
    st = rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, M, N, x.dtype, int(offset), workspace,
                     workspace.numel(), stream)
    if st != RMSNORM_OK:
        raise RMSNormError(st, "rmsnorm_bwd")
    return dx, dgamma


# --------------------------------------------------------------------------- #
# numpy storage arrays <-> device (used by the tests, the smoke check and the bench)
# --------------------------------------------------------------------------- #
TORCH_DTYPES = {"float32": "float32", "float16": "float16", "bfloat16": "bfloat16"}


def to_device(arr, dtype: str, device="cuda"):
    """numpy storage array (float32, or uint16 bit patterns) -> torch CUDA tensor of ``dtype``."""
    import numpy as np
    import torch
    a = np.ascontiguousarray(arr)
    if dtype == "float32":
        return torch.from_numpy(a.astype(np.float32, copy=False)).to(device)
    t = torch.from_numpy(a.view(np.int16)).to(device)
    return t.view(getattr(torch, TORCH_DTYPES[dtype]))


def to_numpy(t, dtype: str):
    """torch tensor -> numpy storage array (float32, or uint16 bit patterns)."""
    import numpy as np
    import torch
    t = t.detach().contiguous().cpu()
    if dtype == "float32" or t.dtype == torch.float32:
        return t.numpy().astype(np.float32, copy=False)
    return t.view(torch.int16).numpy().view(np.uint16)
