"""Torch-facing wrappers over the libnorm C ABI.

These only marshal arguments: they allocate outputs with PyTorch (device
memory plumbing), read pointers, strides and the current CUDA stream, and call
the C entry point of the same name.  Every step of the computation runs in the
library's CUDA kernels; nothing here computes on the CPU or falls back to
PyTorch ops.

Row tensors are (..., H) with the last dim contiguous; the leading dims must
flatten to a single row stride (a view, never a copy).
"""

from __future__ import annotations

import torch

from . import _lib

_DT = {torch.float32: _lib.NORM_F32, torch.bfloat16: _lib.NORM_BF16, torch.float16: _lib.NORM_F16}


def _dtype_code(t: torch.Tensor, what: str) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"{what}: dtype {t.dtype} not supported (float32, bfloat16 or float16)") from None


def _rows(t: torch.Tensor, what: str):
    """(N, H, ld) of a row tensor, as a 2-D view sharing its storage."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dim() < 1:
        raise ValueError(f"{what} must have at least one dim")
    H = t.shape[-1]
    if H > 1 and t.stride(-1) != 1:
        raise ValueError(f"{what}: the last dim must be contiguous")
    try:
        v = t.view(-1, H) if t.dim() != 2 else t
    except RuntimeError:
        raise ValueError(f"{what}: leading dims do not flatten to one row stride") from None
    N = v.shape[0]
    ld = v.stride(0) if N > 1 else max(H, 1)
    return v, N, H, ld


def _vec(t, H, what, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 1 or t.shape[0] != H or \
            (H > 1 and t.stride(0) != 1):
        raise ValueError(f"{what} must be a contiguous CUDA tensor of shape ({H},)")
    if device is not None and t.device != device:
        raise ValueError(f"{what} is on {t.device}, the rows on {device}")
    return t


def _stats(t, N, what, device):
    """A saved statistic: a contiguous fp32 CUDA tensor of N elements (any
    shape, e.g. (B, T) for (B, T, H) rows) on the rows' device."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise ValueError(f"{what} must be float32, not {t.dtype}")
    if t.numel() != N or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous tensor of {N} elements (one per row)")
    if t.device != device:
        raise ValueError(f"{what} is on {t.device}, the rows on {device}")
    return t


def _grad_out(out, ref, N, H, what):
    """The 2-D view of a caller's output tensor, which must match the rows
    (N, H), dtype and device of `ref`."""
    ov, No, Ho, ld = _rows(out, what)
    if (No, Ho) != (N, H) or out.dtype != ref.dtype or out.device != ref.device:
        raise ValueError(f"{what} must match {tuple(ref.shape)} {ref.dtype} on {ref.device} in rows, width, "
                         f"dtype and device")
    return ov, ld


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _w_code(x_code, *params):
    codes = {_DT[p.dtype] for p in params if p is not None}
    if len(codes) > 1:
        raise TypeError("gamma and beta must share a dtype")
    return codes.pop() if codes else x_code


def ln_forward(x, gamma=None, beta=None, eps: float = 1e-5, *, out=None, save_stats: bool = True):
    """LayerNorm over the last dim.  Returns (y, mean, rstd); mean/rstd are
    fp32 of shape (N,) (None when save_stats is False)."""
    xv, N, H, ldx = _rows(x, "x")
    xc = _dtype_code(x, "x")
    gamma, beta = _vec(gamma, H, "gamma", x.device), _vec(beta, H, "beta", x.device)
    wc = _w_code(xc, gamma, beta)
    y = torch.empty_like(x, memory_format=torch.contiguous_format) if out is None else out
    yv, ldy = _grad_out(y, x, N, H, "out")
    mean = torch.empty(N, device=x.device, dtype=torch.float32) if save_stats else None
    rstd = torch.empty(N, device=x.device, dtype=torch.float32) if save_stats else None
    lib = _lib.load()
    with torch.cuda.device(x.device):
        st = lib.ln_forward(xv.data_ptr(), ldx, _ptr(gamma), _ptr(beta), yv.data_ptr(), ldy, _ptr(mean),
                            _ptr(rstd), N, H, float(eps), xc, wc, _stream(x.device))
    _lib.check("ln_forward", st)
    return y, mean, rstd


def rms_forward(x, gamma=None, eps: float = 1e-5, *, out=None, save_stats: bool = True):
    """RMSNorm over the last dim.  Returns (y, rstd)."""
    xv, N, H, ldx = _rows(x, "x")
    xc = _dtype_code(x, "x")
    gamma = _vec(gamma, H, "gamma", x.device)
    wc = _w_code(xc, gamma)
    y = torch.empty_like(x, memory_format=torch.contiguous_format) if out is None else out
    yv, ldy = _grad_out(y, x, N, H, "out")
    rstd = torch.empty(N, device=x.device, dtype=torch.float32) if save_stats else None
    lib = _lib.load()
    with torch.cuda.device(x.device):
        st = lib.rms_forward(xv.data_ptr(), ldx, _ptr(gamma), yv.data_ptr(), ldy, _ptr(rstd), N, H,
                             float(eps), xc, wc, _stream(x.device))
    _lib.check("rms_forward", st)
    return y, rstd


def fused_add_rms_forward(x, residual, gamma=None, eps: float = 1e-6, *, h_out=None, out=None,
                          save_stats: bool = True):
    """h = x + residual (fp32, stored in x's dtype) and y = rmsnorm(h) * gamma.

    ``h_out`` may be a fresh tensor (default), ``x`` or ``residual`` itself
    (in-place update of the residual stream).  Returns (y, h, rstd)."""
    xv, N, H, ldx = _rows(x, "x")
    xc = _dtype_code(x, "x")
    rv, ldr = _grad_out(residual, x, N, H, "residual")
    gamma = _vec(gamma, H, "gamma", x.device)
    wc = _w_code(xc, gamma)
    h = torch.empty_like(x, memory_format=torch.contiguous_format) if h_out is None else h_out
    hv, ldh = _grad_out(h, x, N, H, "h_out")
    y = torch.empty_like(x, memory_format=torch.contiguous_format) if out is None else out
    yv, ldy = _grad_out(y, x, N, H, "out")
    rstd = torch.empty(N, device=x.device, dtype=torch.float32) if save_stats else None
    lib = _lib.load()
    with torch.cuda.device(x.device):
        st = lib.fused_add_rms_forward(xv.data_ptr(), ldx, rv.data_ptr(), ldr, _ptr(gamma), yv.data_ptr(), ldy,
                                       hv.data_ptr(), ldh, _ptr(rstd), N, H, float(eps), xc, wc,
                                       _stream(x.device))
    _lib.check("fused_add_rms_forward", st)
    return y, h, rstd


def bwd_workspace_bytes(H: int, device=None) -> int:
    """Device bytes the backward needs as workspace for row width H."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return int(_lib.load().norm_bwd_workspace_bytes(int(H), dev.index if dev.index is not None else 0))


def _workspace(ws, H, device):
    need = bwd_workspace_bytes(H, device)
    if need == 0:
        raise RuntimeError("could not size the backward workspace (no CUDA device?)")
    if ws is None:
        return torch.empty((need + 3) // 4, device=device, dtype=torch.float32), need
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {device}")
    nbytes = ws.numel() * ws.element_size()
    return ws, nbytes


def ln_backward(dy, x, mean, rstd, gamma=None, *, need_param_grads: bool = True, beta_grad: bool = True,
                workspace=None, dx=None, param_dtype=None):
    """LayerNorm backward.  Returns (dx, dgamma, dbeta) (dgamma/dbeta None when
    need_param_grads is False).  dgamma/dbeta take gamma's dtype (or
    ``param_dtype``, else x's dtype)."""
    xv, N, H, ldx = _rows(x, "x")
    dyv, lddy = _grad_out(dy, x, N, H, "dy")
    xc = _dtype_code(x, "x")
    mean, rstd = _stats(mean, N, "mean", x.device), _stats(rstd, N, "rstd", x.device)
    gamma = _vec(gamma, H, "gamma", x.device)
    wdt = gamma.dtype if gamma is not None else (param_dtype or x.dtype)
    wc = _DT[wdt]
    out = torch.empty_like(x, memory_format=torch.contiguous_format) if dx is None else dx
    ov, lddx = _grad_out(out, x, N, H, "dx")
    dgamma = torch.empty(H, device=x.device, dtype=wdt) if need_param_grads else None
    dbeta = torch.empty(H, device=x.device, dtype=wdt) if (need_param_grads and beta_grad) else None
    ws, wsb = (None, 0)
    if need_param_grads:
        ws, wsb = _workspace(workspace, H, x.device)
    lib = _lib.load()
    with torch.cuda.device(x.device):
        st = lib.ln_backward(dyv.data_ptr(), lddy, xv.data_ptr(), ldx, mean.data_ptr(), rstd.data_ptr(),
                             _ptr(gamma), ov.data_ptr(), lddx, _ptr(dgamma), _ptr(dbeta), _ptr(ws), wsb, N, H,
                             xc, wc, _stream(x.device))
    _lib.check("ln_backward", st)
    return out, dgamma, dbeta


def rms_backward(dy, x, rstd, gamma=None, *, need_param_grads: bool = True, workspace=None, dx=None,
                 param_dtype=None):
    """RMSNorm backward.  Returns (dx, dgamma)."""
    xv, N, H, ldx = _rows(x, "x")
    dyv, lddy = _grad_out(dy, x, N, H, "dy")
    xc = _dtype_code(x, "x")
    rstd = _stats(rstd, N, "rstd", x.device)
    gamma = _vec(gamma, H, "gamma", x.device)
    wdt = gamma.dtype if gamma is not None else (param_dtype or x.dtype)
    wc = _DT[wdt]
    out = torch.empty_like(x, memory_format=torch.contiguous_format) if dx is None else dx
    ov, lddx = _grad_out(out, x, N, H, "dx")
    dgamma = torch.empty(H, device=x.device, dtype=wdt) if need_param_grads else None
    ws, wsb = (None, 0)
    if need_param_grads:
        ws, wsb = _workspace(workspace, H, x.device)
    lib = _lib.load()
    with torch.cuda.device(x.device):
        st = lib.rms_backward(dyv.data_ptr(), lddy, xv.data_ptr(), ldx, rstd.data_ptr(), _ptr(gamma),
                              ov.data_ptr(), lddx, _ptr(dgamma), _ptr(ws), wsb, N, H, xc, wc, _stream(x.device))
    _lib.check("rms_backward", st)
    return out, dgamma


def fused_add_rms_backward(dy, h, rstd, gamma=None, dh_in=None, *, need_param_grads: bool = True,
                           residual_grad: str = "separate", workspace=None, dx=None, param_dtype=None):
    """Backward of fused_add_rms_forward from its stored h and rstd.

    Returns (dx, dres, dgamma): dL/dh for x and for the residual, where
    dL/dh = RMSNorm gradient + dh_in (the gradient arriving through h, or
    None).  ``residual_grad``: "separate" writes a second buffer, "none"
    returns dres = None (the caller reuses dx), "same" treats x and residual
    as one tensor and returns 2 * dL/dh in dx (dres is dx)."""
    hv, N, H, ldh = _rows(h, "h")
    dyv, lddy = _grad_out(dy, h, N, H, "dy")
    xc = _dtype_code(h, "h")
    rstd = _stats(rstd, N, "rstd", h.device)
    gamma = _vec(gamma, H, "gamma", h.device)
    wdt = gamma.dtype if gamma is not None else (param_dtype or h.dtype)
    wc = _DT[wdt]
    if dh_in is not None:
        dv, lddh = _grad_out(dh_in, h, N, H, "dh_in")
    else:
        dv, lddh = None, 0
    out = torch.empty_like(h, memory_format=torch.contiguous_format) if dx is None else dx
    ov, lddx = _grad_out(out, h, N, H, "dx")
    if residual_grad == "separate":
        dres = torch.empty_like(h, memory_format=torch.contiguous_format)
        rv, _, _, lddres = _rows(dres, "dres")
    elif residual_grad == "same":
        dres, rv, lddres = out, ov, lddx
    elif residual_grad == "none":
        dres, rv, lddres = None, None, 0
    else:
        raise ValueError("residual_grad must be 'separate', 'same' or 'none'")
    dgamma = torch.empty(H, device=h.device, dtype=wdt) if need_param_grads else None
    ws, wsb = (None, 0)
    if need_param_grads:
        ws, wsb = _workspace(workspace, H, h.device)
    lib = _lib.load()
    with torch.cuda.device(h.device):
        st = lib.fused_add_rms_backward(dyv.data_ptr(), lddy, hv.data_ptr(), ldh, rstd.data_ptr(), _ptr(gamma),
                                        None if dv is None else dv.data_ptr(), lddh, ov.data_ptr(), lddx,
                                        None if rv is None else rv.data_ptr(), lddres, _ptr(dgamma), _ptr(ws),
                                        wsb, N, H, xc, wc, _stream(h.device))
    _lib.check("fused_add_rms_backward", st)
    return out, (dres if residual_grad == "separate" else (out if residual_grad == "same" else None)), dgamma


def ln_backward_from_output(dy, y, rstd, gamma=None, beta=None, *, need_param_grads: bool = True,
                            beta_grad: bool = True, workspace=None, dx=None, param_dtype=None):
    """LayerNorm backward from the forward's output y (x_hat = (y - beta)/gamma)
    and saved rstd.  Returns (dx, dgamma, dbeta)."""
    yv, N, H, ldy = _rows(y, "y")
    dyv, lddy = _grad_out(dy, y, N, H, "dy")
    xc = _dtype_code(y, "y")
    rstd = _stats(rstd, N, "rstd", y.device)
    gamma, beta = _vec(gamma, H, "gamma", y.device), _vec(beta, H, "beta", y.device)
    wdt = gamma.dtype if gamma is not None else (beta.dtype if beta is not None else (param_dtype or y.dtype))
    wc = _w_code(_DT[wdt], gamma, beta)
    out = torch.empty_like(y, memory_format=torch.contiguous_format) if dx is None else dx
    ov, lddx = _grad_out(out, y, N, H, "dx")
    dgamma = torch.empty(H, device=y.device, dtype=wdt) if need_param_grads else None
    dbeta = torch.empty(H, device=y.device, dtype=wdt) if (need_param_grads and beta_grad) else None
    ws, wsb = (None, 0)
    if need_param_grads:
        ws, wsb = _workspace(workspace, H, y.device)
    lib = _lib.load()
    with torch.cuda.device(y.device):
        st = lib.ln_backward_from_output(dyv.data_ptr(), lddy, yv.data_ptr(), ldy, rstd.data_ptr(), _ptr(gamma),
                                         _ptr(beta), ov.data_ptr(), lddx, _ptr(dgamma), _ptr(dbeta), _ptr(ws), wsb,
                                         N, H, xc, wc, _stream(y.device))
    _lib.check("ln_backward_from_output", st)
    return out, dgamma, dbeta


def rms_backward_from_output(dy, y, rstd, gamma=None, *, need_param_grads: bool = True, workspace=None, dx=None,
                             param_dtype=None):
    """RMSNorm backward from the forward's output y (x_hat = y/gamma) and saved
    rstd.  Returns (dx, dgamma)."""
    yv, N, H, ldy = _rows(y, "y")
    dyv, lddy = _grad_out(dy, y, N, H, "dy")
    xc = _dtype_code(y, "y")
    rstd = _stats(rstd, N, "rstd", y.device)
    gamma = _vec(gamma, H, "gamma", y.device)
    wdt = gamma.dtype if gamma is not None else (param_dtype or y.dtype)
    wc = _DT[wdt]
    out = torch.empty_like(y, memory_format=torch.contiguous_format) if dx is None else dx
    ov, lddx = _grad_out(out, y, N, H, "dx")
    dgamma = torch.empty(H, device=y.device, dtype=wdt) if need_param_grads else None
    ws, wsb = (None, 0)
    if need_param_grads:
        ws, wsb = _workspace(workspace, H, y.device)
    lib = _lib.load()
    with torch.cuda.device(y.device):
        st = lib.rms_backward_from_output(dyv.data_ptr(), lddy, yv.data_ptr(), ldy, rstd.data_ptr(), _ptr(gamma),
                                          ov.data_ptr(), lddx, _ptr(dgamma), _ptr(ws), wsb, N, H, xc, wc,
                                          _stream(y.device))
    _lib.check("rms_backward_from_output", st)
    return out, dgamma
