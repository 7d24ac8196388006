"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle,
compare with the stated tolerances.

Tolerances (the readings of the stated targets):

* fp32 outputs and gradients: max relative error <= 1e-5, measured normwise
  per tensor, max_i |a_i - r_i| / max_i |r_i| (an elementwise ratio is
  undefined where r_i ~ 0).  rstd, never near 0, is checked elementwise; the
  saved mean, often near 0, against the RMS of its row.
* bf16 / fp16 outputs (y, dx): |a_i - r_i| <= ulp(r_i) + 2^-20 * S_i, i.e.
  one ulp of the storage dtype at the exact value plus the fp32 evaluation
  error of the expression, S_i being the magnitude of the terms that are
  summed to form element i.  Equal values (infinities included) pass.
* dgamma/dbeta in bf16 / fp16: relative RMS error ||a - r||_2 / ||r||_2 <= 5e-3.
* the stored residual sum h: bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle as O

F32_TOL = 1e-5
BF16_SLACK = 2.0 ** -20
PARAM_RMS_TOL = 5e-3


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_ulp(r):
    a = np.maximum(np.abs(np.asarray(r, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def f16_ulp(r):
    """Spacing of IEEE binary16 at |r| (10 fraction bits; 2^-24 below 2^-14)."""
    a = np.maximum(np.abs(np.asarray(r, dtype=np.float64)), 2.0 ** -14)
    a = np.where(np.isfinite(a), a, 65504.0)
    return 2.0 ** (np.floor(np.log2(a)) - 10)


def normwise_rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    return num / den if den > 0 else num


def rel_rms(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(np.asarray(got, dtype=np.float64) - ref)
    return num / den if den > 0 else num


def check_f32(got, ref, what, tol=F32_TOL):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e = normwise_rel(got, ref)
    assert e <= tol, f"{what}: normwise relative error {e:.3e} > {tol:.0e}"
    return e


def check_bf16(got, ref, scale, what, ulp=bf16_ulp, allow_inf=False):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if allow_inf:
        assert not np.any(np.isnan(got)), f"{what}: NaN values"
    else:
        assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    with np.errstate(invalid="ignore"):
        err = np.where(got == ref, 0.0, np.abs(got - ref))
    err = np.where(np.isnan(err), np.inf, err)
    tol = ulp(ref) + BF16_SLACK * np.asarray(scale, dtype=np.float64)
    bad = err > tol
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond 1 ulp + fp32 slack; "
                             f"worst at {i}: got {got[i]!r} want {ref[i]!r}")
    strict = int(np.sum(err > ulp(ref)))
    return strict


def check_out(got, ref, scale, dtype, what, allow_inf=False):
    if dtype == torch.float32:
        return check_f32(got, ref, what)
    if dtype == torch.float16:
        return check_bf16(got, ref, scale, what, ulp=f16_ulp, allow_inf=allow_inf)
    return check_bf16(got, ref, scale, what, allow_inf=allow_inf)


DT_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
DT_ORACLE = {torch.float32: "float32", torch.bfloat16: "bfloat16", torch.float16: "float16"}


def check_param(got, ref, dtype, what):
    if dtype == torch.float32:
        return check_f32(got, ref, what)
    e = rel_rms(got, ref)
    assert e <= PARAM_RMS_TOL, f"{what}: relative RMS error {e:.3e} > {PARAM_RMS_TOL:.0e}"
    return e


def check_rstd(got, ref, what):
    rel = np.max(np.abs(got - ref) / np.abs(ref)) if ref.size else 0.0
    assert rel <= F32_TOL, f"{what}: elementwise relative error {rel:.3e}"


def check_mean(got, ref, x, what):
    """The saved mean is checked against the scale of its row, RMS(x_row): a
    mean near 0 has no relative accuracy of its own to speak of."""
    scale = np.sqrt(np.mean(np.asarray(x, dtype=np.float64) ** 2, axis=1))
    rel = np.max(np.abs(got - ref) / np.maximum(scale, 1e-30)) if ref.size else 0.0
    assert rel <= F32_TOL, f"{what}: error relative to the row RMS {rel:.3e}"


# --------------------------------------------------------------------------
# scale terms for the bf16 slack (magnitudes of what is summed per element)
# --------------------------------------------------------------------------

def ln_y_scale(x, mean, rstd, gamma, beta):
    """Magnitude of what y_i = (x_i - mean) * rstd * gamma_i + beta_i is formed
    from.  The fp32 mean carries an absolute error of order eps_fp32 * (|mean|
    + sigma), whatever |x_i - mean| is, so that scale enters x_hat's error."""
    sigma = np.sqrt(np.maximum(1.0 / rstd ** 2, 0.0))
    spread = (np.abs(x - mean[:, None]) + (np.abs(mean) + sigma)[:, None]) * rstd[:, None]
    g = np.ones(x.shape[1]) if gamma is None else gamma
    b = np.zeros(x.shape[1]) if beta is None else beta
    return spread * np.abs(g) + np.abs(b)


def rms_y_scale(x, rstd, gamma):
    g = np.ones(x.shape[1]) if gamma is None else gamma
    return np.abs(x * rstd[:, None] * g)


def ln_dx_scale(dy, x, gamma, eps):
    """Magnitude of what dx_i = rstd * (g_i - c1 - x_hat_i * c2) is formed
    from: x_hat's error scale (|x_i - mean| + |mean| + sigma) * rstd, and the
    row sums c1 = mean(g), c2 = mean(g * x_hat), whose fp32 error scales with
    mean|g| and mean|g * x_hat| rather than with their (cancelling) values."""
    H = x.shape[1]
    g = dy * (np.ones(H) if gamma is None else gamma)
    mean, var = O.two_pass_stats(x)
    r = 1.0 / np.sqrt(var + eps)
    xh = (x - mean[:, None]) * r[:, None]
    spread = (np.abs(x - mean[:, None]) + (np.abs(mean) + np.sqrt(var))[:, None]) * r[:, None]
    c1 = np.abs(g).mean(axis=1, keepdims=True)
    c2 = np.abs(g * xh).mean(axis=1, keepdims=True)
    return r[:, None] * (np.abs(g) + c1 + spread * c2)


def rms_dx_scale(dy, x, gamma, eps):
    """As ln_dx_scale, for dx_i = rstd * (g_i - x_hat_i * c2)."""
    H = x.shape[1]
    g = dy * (np.ones(H) if gamma is None else gamma)
    r = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    xh = x * r[:, None]
    c2 = np.abs(g * xh).mean(axis=1, keepdims=True)
    return r[:, None] * (np.abs(g) + np.abs(xh) * c2)


# --------------------------------------------------------------------------
# guard bands: outputs live inside a larger buffer whose margins must survive
# --------------------------------------------------------------------------

SENTINEL_F32 = 0x7FC0DEAD  # a NaN payload no kernel writes
SENTINEL_BF16 = 0x7FAD


class Guarded:
    """A device tensor of `shape`, with `pad` elements before and after filled
    with a sentinel bit pattern; `ok()` checks the margins are untouched."""

    def __init__(self, shape, dtype, device, pad=64):
        n = int(np.prod(shape)) if len(shape) else 1
        self.dtype = dtype
        self.pad = pad
        ib = torch.int32 if dtype == torch.float32 else torch.int16
        sent = SENTINEL_F32 if dtype == torch.float32 else SENTINEL_BF16
        if ib == torch.int16 and sent >= 2 ** 15:
            sent -= 2 ** 16
        self.raw = torch.full((n + 2 * pad,), sent, dtype=ib, device=device)
        self.sent = sent
        self.t = self.raw.view(dtype)[pad:pad + n].view(*shape)

    def ok(self):
        head = self.raw[:self.pad]
        tail = self.raw[-self.pad:]
        return bool(torch.all(head == self.sent).item() and torch.all(tail == self.sent).item())
