"""GPU-side helpers for the tests: run the C ABI on numpy storage arrays.

Output buffers carry guard regions filled with a sentinel before and after the
data; every run checks the guards afterwards (out-of-bounds writes would show
there). Inputs can be placed one element off a 16-byte boundary to force the
general (scalar) path.
"""
import numpy as np

from rmsnorm_fwd_bwd_gb300 import binding as B

GUARD = 64            # elements of guard before and after each output
SENTINEL = {"float32": np.float32(-12345.5).view(np.uint32), "float16": 0x7BFF, "bfloat16": 0x7F7F}


def _torch():
    import torch
    return torch


def _guarded(n, dtype, device="cuda"):
    """Flat buffer [GUARD + n + GUARD] filled with the sentinel; returns (buffer, view of the n)."""
    torch = _torch()
    if dtype == "float32":
        buf = torch.full((n + 2 * GUARD,), float(np.uint32(SENTINEL[dtype]).view(np.float32)),
                         dtype=torch.float32, device=device)
    else:
        buf = torch.full((n + 2 * GUARD,), int(np.int16(np.uint16(SENTINEL[dtype]).view(np.int16))),
                         dtype=torch.int16, device=device).view(getattr(torch, dtype))
    return buf, buf[GUARD:GUARD + n]


def _guards_intact(buf, dtype):
    a = B.to_numpy(buf, dtype)
    if dtype == "float32":
        a = a.view(np.uint32)
    s = SENTINEL[dtype]
    return bool(np.all(a[:GUARD] == s) and np.all(a[-GUARD:] == s))


def _place(arr, dtype, misalign):
    torch = _torch()
    t = B.to_device(arr.reshape(-1), dtype)
    if not misalign:
        return t, t
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    buf[1:] = t
    return buf, buf[1:]


def run(x, g, dy, dtype, offset=False, eps=1e-6, misalign=False, do_bwd=True, stream=None, ws_fill=None,
        ws_bytes=None):
    """Forward (and backward) through the C ABI. Returns numpy storage arrays
    (y, rstd, dx, dgamma); dx/dgamma are None when do_bwd is False.

    misalign: False, True (every tensor one element off a 16-byte boundary) or a
    set of names among {"x", "g", "dy", "y", "dx"} to shift only those.
    ws_fill: None (the workspace as torch.empty leaves it), a byte value, or
    "random" (seeded random bytes); ws_bytes: the workspace size passed to the
    backward (default: rmsnorm_bwd_workspace_size)."""
    torch = _torch()
    M, N = x.shape
    names = {"x", "g", "dy", "y", "dx"} if misalign is True else set(misalign or ())
    keep = []
    _, xt = _place(x, dtype, "x" in names); keep.append(_)
    _, gt = _place(g, dtype, "g" in names); keep.append(_)
    _, dyt = _place(dy, dtype, "dy" in names); keep.append(_)
    ybuf, y = _guarded(M * N, dtype)
    rbuf, rstd = _guarded(M, "float32")
    if "y" in names:
        ybuf2 = torch.empty(M * N + 2 * GUARD + 1, dtype=y.dtype, device=y.device)
        ybuf2[1:] = ybuf
        ybuf, y = ybuf2[1:], ybuf2[1 + GUARD:1 + GUARD + M * N]
    st = B.rmsnorm_fwd(xt, gt, y, rstd, M, N, eps, dtype, int(offset), stream)
    assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)
    dx = dg = None
    dxbuf = dgbuf = None
    if do_bwd:
        dxbuf, dxt = _guarded(M * N, dtype)
        dgbuf, dgt = _guarded(N, dtype)
        if "dx" in names:
            b2 = torch.empty(M * N + 2 * GUARD + 1, dtype=dxt.dtype, device=dxt.device)
            b2[1:] = dxbuf
            dxbuf, dxt = b2[1:], b2[1 + GUARD:1 + GUARD + M * N]
        wsz = B.rmsnorm_bwd_workspace_size(M, N, dtype) if ws_bytes is None else int(ws_bytes)
        ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device="cuda")
        if ws_fill == "random":
            gen = torch.Generator(device="cuda").manual_seed(1234)
            ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda", generator=gen))
        elif ws_fill is not None:
            ws.fill_(int(ws_fill))
        st = B.rmsnorm_bwd(dyt, xt, gt, rstd, dxt, dgt, M, N, dtype, int(offset), ws, wsz, stream)
        assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)
    torch.cuda.synchronize()
    assert _guards_intact(ybuf, dtype), "forward wrote outside y"
    assert _guards_intact(rbuf, "float32"), "forward wrote outside rstd"
    yo = B.to_numpy(y, dtype).reshape(M, N)
    ro = B.to_numpy(rstd, "float32")
    if do_bwd:
        assert _guards_intact(dxbuf, dtype), "backward wrote outside dx"
        assert _guards_intact(dgbuf, dtype), "backward wrote outside dgamma"
        dx = B.to_numpy(dxt, dtype).reshape(M, N)
        dg = B.to_numpy(dgt, dtype)
    return yo, ro, dx, dg


def ln_run(x, g, b, dy, dtype, eps=1e-5, misalign=False, do_bwd=True, stats=True, stream=None):
    """LayerNorm forward (and backward) through the C ABI, dense rows. Returns
    numpy storage arrays (y, mean, rstd, dx, dgamma, dbeta); mean and rstd are
    None when ``stats`` is False (the forward is then called with NULL for
    them), the gradients None when ``do_bwd`` is False.

    misalign: False, True, or a set of names among {"x", "g", "b", "dy", "y", "dx"}."""
    torch = _torch()
    M, N = x.shape
    names = {"x", "g", "b", "dy", "y", "dx"} if misalign is True else set(misalign or ())
    keep = []
    _, xt = _place(x, dtype, "x" in names); keep.append(_)
    _, gt = _place(g, dtype, "g" in names); keep.append(_)
    _, bt = _place(b, dtype, "b" in names); keep.append(_)
    _, dyt = _place(dy, dtype, "dy" in names); keep.append(_)

    def out(n, name):
        buf, view = _guarded(n, dtype)
        if name in names:
            b2 = torch.empty(n + 2 * GUARD + 1, dtype=view.dtype, device=view.device)
            b2[1:] = buf
            buf, view = b2[1:], b2[1 + GUARD:1 + GUARD + n]
        return buf, view

    ybuf, y = out(M * N, "y")
    mbuf, mean = _guarded(M, "float32")
    rbuf, rstd = _guarded(M, "float32")
    st = B.layernorm_fwd(xt, N, gt, bt, y, N, mean if stats else None, rstd if stats else None, M, N, eps,
                         dtype, stream)
    assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)
    res = [None] * 6
    if do_bwd:
        if not stats:
            raise ValueError("the backward needs the saved statistics")
        dxbuf, dxt = out(M * N, "dx")
        dgbuf, dgt = _guarded(N, dtype)
        dbbuf, dbt = _guarded(N, dtype)
        wsz = B.layernorm_bwd_workspace_size(M, N, dtype)
        ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device="cuda")
        st = B.layernorm_bwd(dyt, N, xt, N, gt, mean, rstd, dxt, N, dgt, dbt, M, N, dtype, ws, wsz, stream)
        assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)
    torch.cuda.synchronize()
    assert _guards_intact(ybuf, dtype), "forward wrote outside y"
    assert _guards_intact(mbuf, "float32"), "forward wrote outside mean"
    assert _guards_intact(rbuf, "float32"), "forward wrote outside rstd"
    res[0] = B.to_numpy(y, dtype).reshape(M, N)
    if stats:
        res[1] = B.to_numpy(mean, "float32")
        res[2] = B.to_numpy(rstd, "float32")
    else:
        sent = np.uint32(SENTINEL["float32"]).view(np.float32)
        assert np.all(B.to_numpy(mean, "float32") == sent) and np.all(B.to_numpy(rstd, "float32") == sent), \
            "forward wrote mean/rstd although they were NULL"
    if do_bwd:
        assert _guards_intact(dxbuf, dtype), "backward wrote outside dx"
        assert _guards_intact(dgbuf, dtype), "backward wrote outside dgamma"
        assert _guards_intact(dbbuf, dtype), "backward wrote outside dbeta"
        res[3] = B.to_numpy(dxt, dtype).reshape(M, N)
        res[4] = B.to_numpy(dgt, dtype)
        res[5] = B.to_numpy(dbt, dtype)
    return tuple(res)


def dbwd_run(ddx, ddg, dy, x, g, dtype, offset=False, eps=1e-6, misalign=False, stream=None):
    """RMSNorm forward (for r) then the double backward through the C ABI, dense
    rows. ddg may be None. Returns numpy storage arrays (d_dy, d_x, d_gamma).

    misalign: False, True, or a set of names among {"ddx", "dy", "x", "d_dy", "d_x"}."""
    torch = _torch()
    M, N = x.shape
    names = {"ddx", "dy", "x", "d_dy", "d_x"} if misalign is True else set(misalign or ())
    keep = []
    _, xt = _place(x, dtype, "x" in names); keep.append(_)
    _, gt = _place(g, dtype, False); keep.append(_)
    _, dyt = _place(dy, dtype, "dy" in names); keep.append(_)
    _, tt = _place(ddx, dtype, "ddx" in names); keep.append(_)
    qt = None
    if ddg is not None:
        _, qt = _place(ddg, dtype, False); keep.append(_)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    y = torch.empty(M * N, dtype=xt.dtype, device="cuda")
    st = B.rmsnorm_fwd(xt, gt, y, rstd, M, N, eps, dtype, int(offset), stream)
    assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)

    def out(n, name):
        buf, view = _guarded(n, dtype)
        if name in names:
            b2 = torch.empty(n + 2 * GUARD + 1, dtype=view.dtype, device=view.device)
            b2[1:] = buf
            buf, view = b2[1:], b2[1 + GUARD:1 + GUARD + n]
        return buf, view

    odybuf, ody = out(M * N, "d_dy")
    oxbuf, ox = out(M * N, "d_x")
    ogbuf, og = _guarded(N, dtype)
    wsz = B.rmsnorm_bwd_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device="cuda")
    st = B.rmsnorm_bwd_bwd(tt, N, qt, dyt, N, xt, N, gt, rstd, ody, N, ox, N, og, M, N, dtype, int(offset),
                           ws, wsz, stream)
    assert st == B.RMSNORM_OK, B.rmsnorm_status_string(st)
    torch.cuda.synchronize()
    assert _guards_intact(odybuf, dtype), "double backward wrote outside d_dy"
    assert _guards_intact(oxbuf, dtype), "double backward wrote outside d_x"
    assert _guards_intact(ogbuf, dtype), "double backward wrote outside d_gamma"
    return (B.to_numpy(ody, dtype).reshape(M, N), B.to_numpy(ox, dtype).reshape(M, N), B.to_numpy(og, dtype))
