"""PyTorch integration of the C-ABI kernels: autograd and torch.library ops.

``rms_norm(x, weight, eps, offset)`` runs the library's forward kernel and, in
the backward pass, its fused backward kernels -- the calls
``binding.rmsnorm_fwd_strided`` / ``binding.rmsnorm_bwd_strided``, with tensors
allocated by torch. 2-D inputs whose rows are further apart than their length
(e.g. ``big[:, :N]``) are passed with their row pitch, without a copy. It is
registered as the custom ops ``rmsnorm_gb300::fwd`` and ``rmsnorm_gb300::bwd``
(with fake-tensor shapes and an autograd formula), so it traces without graph
breaks.

Mirrors the autograd adapter of the page "Check an AI model calculation before
accelerating it" (section "Connecting Autograd and actually training"): the
forward saves x, gamma and the per-row r; the backward returns dx and dgamma and
nothing for eps; ``CALLS`` counts passes through the adapter so a training loop
can prove it ran the kernel path.

``layer_norm(x, weight, bias, eps)`` does the same for LayerNorm through
``binding.layernorm_fwd`` / ``binding.layernorm_bwd`` (custom ops
``rmsnorm_gb300::ln_fwd`` / ``rmsnorm_gb300::ln_bwd``): the forward saves x,
gamma and the per-row mean and r; the backward returns dx, dgamma and dbeta.
``LN_CALLS`` counts its passes.

The backward op has an autograd formula of its own (double backward): the
gradients of sum(ddx * dx) + sum(ddw * dw) for dy, x and the weight come from
``binding.rmsnorm_bwd_bwd`` (custom op ``rmsnorm_gb300::bwd_bwd``), so
``torch.autograd.grad(..., create_graph=True)`` through ``rms_norm`` runs on the
library's kernels at both orders. ``CALLS["double_backward"]`` counts them.
"""
from __future__ import annotations

import os

import torch

from . import binding

CALLS = {"forward": 0, "backward": 0, "double_backward": 0}
LN_CALLS = {"forward": 0, "backward": 0}

# A kernel whose bounded wait gives up returns early with its outputs partly
# unwritten and reports it only through the device error word (the host call
# itself succeeded). RMSNORM_CHECK_DEVICE_ERROR=1 reads that word after every op
# (a device synchronisation each time) and raises; otherwise call
# check_device_error() at the end of a training step.
CHECK_EVERY_OP = os.environ.get("RMSNORM_CHECK_DEVICE_ERROR", "0") not in ("", "0")


class DeviceError(RuntimeError):
    """A kernel reported a failure through the device error word."""


def check_device_error(clear: bool = True) -> None:
    """Raise DeviceError if any kernel on the current device has set the device
    error word since it was last cleared (bit 0: a bounded wait gave up; bit 1,
    debug builds: a read outside its tensor). Synchronizes the device."""
    word = binding.rmsnorm_device_error(clear=clear)
    if word:
        raise DeviceError(f"RMSNorm kernels reported device error word {word:#x}")


def _after_op():
    if CHECK_EVERY_OP:
        check_device_error()


def _rows(x: torch.Tensor):
    N = x.shape[-1]
    return (x.numel() // N if N else 0), N


def _row_view(t: torch.Tensor):
    """(tensor, row pitch): 2-D views with unit column stride keep their row
    pitch (no copy); anything else is made contiguous."""
    if t.dim() == 2 and t.stride(1) == 1 and t.stride(0) >= t.shape[1] and t.shape[0] > 0:
        return t, t.stride(0)
    t = t.contiguous()
    return t, t.shape[-1]


@torch.library.custom_op("rmsnorm_gb300::fwd", mutates_args=())
def _fwd(x: torch.Tensor, weight: torch.Tensor, eps: float, offset: bool) -> tuple[torch.Tensor, torch.Tensor]:
    x, ldx = _row_view(x)
    M, N = _rows(x)
    y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = binding.rmsnorm_fwd_strided(x, ldx, weight.contiguous(), y, N, rstd, M, N, eps, x.dtype,
                                     int(offset), torch.cuda.current_stream(x.device))
    if st != binding.RMSNORM_OK:
        raise binding.RMSNormError(st, "rmsnorm_fwd")
    CALLS["forward"] += 1
    _after_op()
    return y, rstd


@_fwd.register_fake
def _(x, weight, eps, offset):
    return x.new_empty(x.shape), x.new_empty(x.shape[:-1], dtype=torch.float32)


@torch.library.custom_op("rmsnorm_gb300::bwd", mutates_args=())
def _bwd(dy: torch.Tensor, x: torch.Tensor, weight: torch.Tensor, rstd: torch.Tensor,
         offset: bool) -> tuple[torch.Tensor, torch.Tensor]:
    dy, lddy = _row_view(dy)
    x, ldx = _row_view(x)
    M, N = _rows(x)
    need = binding.rmsnorm_bwd_workspace_size(M, N, x.dtype)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    dx = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    dw = torch.empty(weight.shape, dtype=weight.dtype, device=weight.device)
    st = binding.rmsnorm_bwd_strided(dy, lddy, x, ldx, weight.contiguous(), rstd.contiguous(), dx, N, dw, M, N,
                                     x.dtype, int(offset), ws, ws.numel(), torch.cuda.current_stream(x.device))
    if st != binding.RMSNORM_OK:
        raise binding.RMSNormError(st, "rmsnorm_bwd")
    CALLS["backward"] += 1
    _after_op()
    return dx, dw


@_bwd.register_fake
def _(dy, x, weight, rstd, offset):
    return x.new_empty(x.shape), weight.new_empty(weight.shape)


def _setup_context(ctx, inputs, output):
    x, weight, eps, offset = inputs
    _, rstd = output
    ctx.save_for_backward(x, weight, rstd)
    ctx.offset = offset


def _backward(ctx, dy, drstd):
    del drstd  # rstd is an auxiliary output; no gradient flows through it
    x, weight, rstd = ctx.saved_tensors
    dx, dw = _bwd(dy, x, weight, rstd, ctx.offset)
    return dx, dw, None, None


_fwd.register_autograd(_backward, setup_context=_setup_context)


@torch.library.custom_op("rmsnorm_gb300::bwd_bwd", mutates_args=())
def _bwd_bwd(ddx: torch.Tensor, ddw: torch.Tensor, dy: torch.Tensor, x: torch.Tensor, weight: torch.Tensor,
             rstd: torch.Tensor, offset: bool) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    ddx, ldt = _row_view(ddx)
    dy, lddy = _row_view(dy)
    x, ldx = _row_view(x)
    M, N = _rows(x)
    need = binding.rmsnorm_bwd_bwd_workspace_size(M, N, x.dtype)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    d_dy = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    d_x = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    d_w = torch.empty(weight.shape, dtype=weight.dtype, device=weight.device)
    st = binding.rmsnorm_bwd_bwd(ddx, ldt, ddw.contiguous(), dy, lddy, x, ldx, weight.contiguous(),
                                 rstd.contiguous(), d_dy, N, d_x, N, d_w, M, N, x.dtype, int(offset), ws,
                                 ws.numel(), torch.cuda.current_stream(x.device))
    if st != binding.RMSNORM_OK:
        raise binding.RMSNormError(st, "rmsnorm_bwd_bwd")
    CALLS["double_backward"] += 1
    _after_op()
    return d_dy, d_x, d_w


@_bwd_bwd.register_fake
def _(ddx, ddw, dy, x, weight, rstd, offset):
    return x.new_empty(x.shape), x.new_empty(x.shape), weight.new_empty(weight.shape)


def _bwd_setup_context(ctx, inputs, output):
    dy, x, weight, rstd, offset = inputs
    ctx.save_for_backward(dy, x, weight, rstd)
    ctx.offset = offset


def _bwd_backward(ctx, ddx, ddw):
    dy, x, weight, rstd = ctx.saved_tensors
    if ddx is None:
        ddx = torch.zeros_like(x)
    if ddw is None:
        ddw = torch.zeros_like(weight)
    d_dy, d_x, d_w = _bwd_bwd(ddx, ddw, dy, x, weight, rstd, ctx.offset)
    # rstd is a function of x; its dependence is already inside d_x
    return d_dy, d_x, d_w, None, None


_bwd.register_autograd(_bwd_backward, setup_context=_bwd_setup_context)


def rms_norm(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6, offset: bool = False) -> torch.Tensor:
    """y = x * r * weight (offset: x * r * (1 + weight)), r = 1/sqrt(mean(x^2, -1) + eps)."""
    if x.shape[-1] != weight.shape[-1] or weight.dim() != 1:
        raise ValueError("weight must be 1-D with x.shape[-1] elements")
    if x.dtype != weight.dtype:
        raise ValueError("x and weight must share a dtype")
    y, _ = torch.ops.rmsnorm_gb300.fwd(x, weight, float(eps), bool(offset))
    return y


class RMSNorm(torch.nn.Module):
    """Drop-in module: a learned weight of ``normalized_shape`` elements (ones,
    or zeros for the offset variant, so that both start as the identity scale)."""

    def __init__(self, normalized_shape: int, eps: float = 1e-6, offset: bool = False,
                 device=None, dtype=None):
        super().__init__()
        self.eps = eps
        self.offset = offset
        init = torch.zeros if offset else torch.ones
        self.weight = torch.nn.Parameter(init(normalized_shape, device=device, dtype=dtype))

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return rms_norm(x, self.weight, self.eps, self.offset)


# --------------------------------------------------------------------------- #
# LayerNorm
# --------------------------------------------------------------------------- #
@torch.library.custom_op("rmsnorm_gb300::ln_fwd", mutates_args=())
def _ln_fwd(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor,
            eps: float) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    x, ldx = _row_view(x)
    M, N = _rows(x)
    y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    st = binding.layernorm_fwd(x, ldx, weight.contiguous(), bias.contiguous(), y, N, mean, rstd, M, N, eps,
                               x.dtype, torch.cuda.current_stream(x.device))
    if st != binding.RMSNORM_OK:
        raise binding.RMSNormError(st, "layernorm_fwd")
    LN_CALLS["forward"] += 1
    _after_op()
    return y, mean, rstd


@_ln_fwd.register_fake
def _(x, weight, bias, eps):
    return (x.new_empty(x.shape), x.new_empty(x.shape[:-1], dtype=torch.float32),
            x.new_empty(x.shape[:-1], dtype=torch.float32))


@torch.library.custom_op("rmsnorm_gb300::ln_bwd", mutates_args=())
def _ln_bwd(dy: torch.Tensor, x: torch.Tensor, weight: torch.Tensor, mean: torch.Tensor,
            rstd: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    dy, lddy = _row_view(dy)
    x, ldx = _row_view(x)
    M, N = _rows(x)
    need = binding.layernorm_bwd_workspace_size(M, N, x.dtype)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    dx = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    dw = torch.empty(weight.shape, dtype=weight.dtype, device=weight.device)
    db = torch.empty(weight.shape, dtype=weight.dtype, device=weight.device)
    st = binding.layernorm_bwd(dy, lddy, x, ldx, weight.contiguous(), mean.contiguous(), rstd.contiguous(),
                               dx, N, dw, db, M, N, x.dtype, ws, ws.numel(), torch.cuda.current_stream(x.device))
    if st != binding.RMSNORM_OK:
        raise binding.RMSNormError(st, "layernorm_bwd")
    LN_CALLS["backward"] += 1
    _after_op()
    return dx, dw, db


@_ln_bwd.register_fake
def _(dy, x, weight, mean, rstd):
    return x.new_empty(x.shape), weight.new_empty(weight.shape), weight.new_empty(weight.shape)


def _ln_setup_context(ctx, inputs, output):
    x, weight, _bias, _eps = inputs
    _, mean, rstd = output
    ctx.save_for_backward(x, weight, mean, rstd)


def _ln_backward(ctx, dy, dmean, drstd):
    del dmean, drstd  # auxiliary outputs; no gradient flows through them
    x, weight, mean, rstd = ctx.saved_tensors
    dx, dw, db = _ln_bwd(dy, x, weight, mean, rstd)
    return dx, dw, db, None


_ln_fwd.register_autograd(_ln_backward, setup_context=_ln_setup_context)


def layer_norm(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor, eps: float = 1e-5) -> torch.Tensor:
    """y = (x - mean) * r * weight + bias over the last dimension,
    r = 1/sqrt(biased variance + eps)."""
    N = x.shape[-1]
    for name, t in (("weight", weight), ("bias", bias)):
        if t.dim() != 1 or t.shape[0] != N:
            raise ValueError(f"{name} must be 1-D with x.shape[-1] elements")
        if t.dtype != x.dtype:
            raise ValueError(f"x and {name} must share a dtype")
    y, _, _ = torch.ops.rmsnorm_gb300.ln_fwd(x, weight, bias, float(eps))
    return y


class LayerNorm(torch.nn.Module):
    """Drop-in module with a learned weight (ones) and bias (zeros) of
    ``normalized_shape`` elements."""

    def __init__(self, normalized_shape: int, eps: float = 1e-5, device=None, dtype=None):
        super().__init__()
        self.eps = eps
        self.weight = torch.nn.Parameter(torch.ones(normalized_shape, device=device, dtype=dtype))
        self.bias = torch.nn.Parameter(torch.zeros(normalized_shape, device=device, dtype=dtype))

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return layer_norm(x, self.weight, self.bias, self.eps)
