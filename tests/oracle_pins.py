"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes a namespace ``O`` holding the oracle's functions, so that
``test_oracle_mutants.py`` can run the same pins against copies of the oracle
with a planted mistake and show that every such mistake is caught.

What pins what:

* torch's CPU fp64 ``layer_norm`` / ``rms_norm`` and autograd (library
  routines written independently of the oracle) -- forward and backward;
* central finite differences of the oracle's own forward -- every backward;
* invariants of the mathematics: shift and scale behaviour of the normalised
  row, the LayerNorm grad_input summing to zero along a row, and the
  homogeneity identities derived in the docstrings below;
* closed forms: H = 1, constant rows, two-element rows;
* Welford's recurrence and the parallel merge against the two-pass
  definition and numpy's mean/var;
* the bfloat16 rounding helper against torch's own cast.
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _rng(seed):
    return np.random.default_rng(seed)


def _case(seed, N, H, offset=0.0):
    r = _rng(seed)
    x = offset + r.standard_normal((N, H))
    gamma = 1.0 + 0.1 * r.standard_normal(H)
    beta = 0.1 * r.standard_normal(H)
    dy = r.standard_normal((N, H))
    res = r.standard_normal((N, H))
    return x, gamma, beta, dy, res


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    tol = atol + rtol * np.abs(b)
    bad = err > tol
    assert not np.any(bad), f"{what}: max abs err {err.max():.3e} (worst at {np.unravel_index(np.argmax(err - tol), err.shape)})"


SHAPES = [(3, 7), (2, 33), (5, 256), (4, 1), (2, 2), (7, 1000)]


# --------------------------------------------------------------------------
# library cross-checks (torch CPU float64)
# --------------------------------------------------------------------------

def pin_ln_forward_vs_torch(O):
    for i, (N, H) in enumerate(SHAPES):
        for eps in (1e-5, 1e-2):
            x, gamma, beta, _, _ = _case(10 + i, N, H)
            y, mean, rstd = O.layer_norm_forward(x, gamma, beta, eps)
            yt = F.layer_norm(torch.from_numpy(x), (H,), torch.from_numpy(gamma),
                              torch.from_numpy(beta), eps).numpy()
            _close(y, yt, 1e-12, 1e-12, f"ln y {N}x{H}")
            _close(mean, x.mean(axis=1), 1e-12, 1e-12, "ln mean")
            _close(rstd, 1.0 / np.sqrt(x.var(axis=1) + eps), 1e-12, 0, "ln rstd")


def pin_rms_forward_vs_torch(O):
    for i, (N, H) in enumerate(SHAPES):
        for eps in (1e-6, 1e-2):
            x, gamma, _, _, _ = _case(20 + i, N, H)
            y, rstd = O.rms_norm_forward(x, gamma, eps)
            yt = F.rms_norm(torch.from_numpy(x), (H,), torch.from_numpy(gamma), eps).numpy()
            _close(y, yt, 1e-12, 1e-12, f"rms y {N}x{H}")
            _close(rstd, 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps), 1e-12, 0, "rms rstd")


def _autograd(fn, x, gamma, beta, dy):
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    gt = torch.from_numpy(gamma.copy()).requires_grad_(True)
    bt = None if beta is None else torch.from_numpy(beta.copy()).requires_grad_(True)
    y = fn(xt, gt, bt)
    y.backward(torch.from_numpy(dy))
    return xt.grad.numpy(), gt.grad.numpy(), (None if bt is None else bt.grad.numpy())


def pin_ln_backward_vs_autograd(O):
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-5
        x, gamma, beta, dy, _ = _case(30 + i, N, H)
        dx, dg, db = O.layer_norm_backward(dy, x, gamma, eps)
        tdx, tdg, tdb = _autograd(lambda a, g, b: F.layer_norm(a, (H,), g, b, eps), x, gamma, beta, dy)
        _close(dx, tdx, 1e-9, 1e-11, f"ln dx {N}x{H}")
        _close(dg, tdg, 1e-9, 1e-11, "ln dgamma")
        _close(db, tdb, 1e-12, 1e-12, "ln dbeta")


def pin_rms_backward_vs_autograd(O):
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-6
        x, gamma, _, dy, _ = _case(40 + i, N, H)
        dx, dg = O.rms_norm_backward(dy, x, gamma, eps)
        tdx, tdg, _ = _autograd(lambda a, g, b: F.rms_norm(a, (H,), g, eps), x, gamma, None, dy)
        _close(dx, tdx, 1e-9, 1e-11, f"rms dx {N}x{H}")
        _close(dg, tdg, 1e-9, 1e-11, "rms dgamma")


# --------------------------------------------------------------------------
# central finite differences of the oracle's own forward
# --------------------------------------------------------------------------

def _fd(loss, arr, step=1e-6):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        keep = arr[idx]
        arr[idx] = keep + step
        lp = loss()
        arr[idx] = keep - step
        lm = loss()
        arr[idx] = keep
        g[idx] = (lp - lm) / (2 * step)
    return g


FD_SHAPES = [(3, 7), (2, 33), (1, 1), (2, 2)]


def pin_fd_layer_norm(O):
    for i, (N, H) in enumerate(FD_SHAPES):
        eps = 1e-3
        x, gamma, beta, w, _ = _case(50 + i, N, H)
        loss = lambda: float(np.sum(w * O.layer_norm_forward(x, gamma, beta, eps)[0]))
        dx, dg, db = O.layer_norm_backward(w, x, gamma, eps)
        _close(dx, _fd(loss, x), 1e-6, 1e-7, f"fd ln dx {N}x{H}")
        _close(dg, _fd(loss, gamma), 1e-6, 1e-7, "fd ln dgamma")
        _close(db, _fd(loss, beta), 1e-6, 1e-7, "fd ln dbeta")


def pin_fd_rms_norm(O):
    for i, (N, H) in enumerate(FD_SHAPES):
        eps = 1e-3
        x, gamma, _, w, _ = _case(60 + i, N, H)
        loss = lambda: float(np.sum(w * O.rms_norm_forward(x, gamma, eps)[0]))
        dx, dg = O.rms_norm_backward(w, x, gamma, eps)
        _close(dx, _fd(loss, x), 1e-6, 1e-7, f"fd rms dx {N}x{H}")
        _close(dg, _fd(loss, gamma), 1e-6, 1e-7, "fd rms dgamma")


def pin_fd_fused(O):
    for i, (N, H) in enumerate(FD_SHAPES):
        eps = 1e-3
        x, gamma, _, w, res = _case(70 + i, N, H)
        loss = lambda: float(np.sum(w * O.fused_add_rms_norm_forward(x, res, gamma, eps, "float64")[0]))
        dx, dres, dg = O.fused_add_rms_norm_backward(w, x, res, gamma, eps)
        _close(dx, _fd(loss, x), 1e-6, 1e-7, f"fd fused dx {N}x{H}")
        _close(dres, _fd(loss, res), 1e-6, 1e-7, "fd fused dres")
        _close(dg, _fd(loss, gamma), 1e-6, 1e-7, "fd fused dgamma")


# --------------------------------------------------------------------------
# invariants of the mathematics
# --------------------------------------------------------------------------

def pin_ln_invariants(O):
    """LayerNorm identities.

    * With gamma = 1, beta = 0 the output is x_hat: every row has mean 0 and
      mean(x_hat^2) = var/(var + eps), var taken from numpy.
    * y(c*x + s) with eps scaled by c^2 equals y(x): shift and scale invariance.
    * Shift invariance of the loss gives sum_j dx_j = 0 on every row.
    * Scale: d/dc L(mu + c*(x - mu)) at c = 1 equals sum_j (x_j - mu) dx_j; as
      x_hat(c) = c*(x-mu)/sqrt(c^2 var + eps), this is
      rstd * eps/(var + eps) * sum_j (x_j - mu) g_j  with g = dy*gamma.
    * dbeta is the column sum of dy; dgamma is the column sum of dy * x_hat
      with x_hat read back from a gamma=1, beta=0 forward.
    """
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-3
        x, gamma, beta, dy, _ = _case(80 + i, N, H, offset=3.0)
        xhat = O.layer_norm_forward(x, None, None, eps)[0]
        var = x.var(axis=1)
        _close(xhat.mean(axis=1), np.zeros(N), 0, 1e-12, "mean(x_hat)")
        _close((xhat * xhat).mean(axis=1), var / (var + eps), 1e-12, 1e-15, "mean(x_hat^2)")
        c, s = 3.5, -2.25
        y1 = O.layer_norm_forward(x, gamma, beta, eps)[0]
        y2 = O.layer_norm_forward(c * x + s, gamma, beta, eps * c * c)[0]
        _close(y2, y1, 1e-11, 1e-11, "ln affine invariance")
        dx, dg, db = O.layer_norm_backward(dy, x, gamma, eps)
        _close(dx.sum(axis=1), np.zeros(N), 0, 1e-10, "sum(dx)")
        mu = x.mean(axis=1, keepdims=True)
        rstd = 1.0 / np.sqrt(var + eps)
        lhs = ((x - mu) * dx).sum(axis=1)
        rhs = rstd * eps / (var + eps) * ((x - mu) * dy * gamma).sum(axis=1)
        _close(lhs, rhs, 1e-9, 1e-11, "ln scale identity")
        _close(db, dy.sum(axis=0), 1e-13, 1e-13, "dbeta")
        _close(dg, (dy * xhat).sum(axis=0), 1e-12, 1e-12, "dgamma")


def pin_rms_invariants(O):
    """RMSNorm identities.

    * gamma = 1: mean(y^2) = m/(m + eps) with m = mean(x^2) from numpy.
    * y(c*x) with eps scaled by c^2 equals y(x).
    * Scale: sum_j x_j dx_j = rstd * eps/(m + eps) * sum_j x_j g_j.
    * dgamma is the column sum of dy * y(gamma=1).
    """
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-3
        x, gamma, _, dy, _ = _case(90 + i, N, H, offset=0.5)
        y1 = O.rms_norm_forward(x, None, eps)[0]
        m = np.mean(x * x, axis=1)
        _close((y1 * y1).mean(axis=1), m / (m + eps), 1e-12, 1e-15, "mean(y^2)")
        c = -2.75
        _close(O.rms_norm_forward(c * x, gamma, eps * c * c)[0],
               O.rms_norm_forward(x, gamma, eps)[0] * np.sign(c), 1e-11, 1e-11, "rms scale invariance")
        dx, dg = O.rms_norm_backward(dy, x, gamma, eps)
        rstd = 1.0 / np.sqrt(m + eps)
        _close((x * dx).sum(axis=1), rstd * eps / (m + eps) * (x * dy * gamma).sum(axis=1),
               1e-9, 1e-11, "rms scale identity")
        _close(dg, (dy * y1).sum(axis=0), 1e-12, 1e-12, "rms dgamma")


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def pin_closed_forms(O):
    """Cases whose answers are known without the general formula.

    * Constant rows (zero variance, including H = 1): LayerNorm gives y = beta,
      mean = the constant, rstd = eps^-1/2.  The variance is flat there
      (d var/dx = 2(x - mean)/H = 0), so dy_j/dx_k = (delta_jk - 1/H) rstd gamma_j
      and dx = eps^-1/2 * (g - mean(g)) with g = dy*gamma; dgamma = 0.
    * Two-element rows [a, b]: x_hat = +-d / sqrt(d^2 + eps) with d = (a-b)/2.
    * RMSNorm of a constant row c: y = gamma * c / sqrt(c^2 + eps).
    * LayerNorm with gamma = 1, beta = 0 on a row of N(mu, s^2)-like data
      reduces to the textbook standard score (x - mean)/sqrt(var + eps).
    """
    eps = 1e-5
    beta = np.array([0.25, -1.5, 3.0])
    gamma = np.array([2.0, 0.5, -1.0])
    x = np.array([[4.0, 4.0, 4.0], [-7.5, -7.5, -7.5]])
    y, mean, rstd = O.layer_norm_forward(x, gamma, beta, eps)
    _close(y, np.tile(beta, (2, 1)), 0, 0, "const-row y")
    _close(mean, [4.0, -7.5], 0, 0, "const-row mean")
    _close(rstd, [eps ** -0.5] * 2, 1e-15, 0, "const-row rstd")
    dy = np.array([[1.0, -2.0, 0.5], [0.3, 0.7, -1.1]])
    dx, dg, db = O.layer_norm_backward(dy, x, gamma, eps)
    g = dy * gamma
    _close(dx, eps ** -0.5 * (g - g.mean(axis=1, keepdims=True)), 1e-12, 1e-12, "const-row dx")
    _close(dg, np.zeros(3), 0, 1e-12, "const-row dgamma")
    _close(db, dy.sum(axis=0), 0, 1e-15, "const-row dbeta")

    x1 = np.array([[3.0], [-2.0], [0.0]])
    y1, m1, r1 = O.layer_norm_forward(x1, np.array([5.0]), np.array([0.75]), eps)
    _close(y1, np.full((3, 1), 0.75), 0, 0, "H=1 y")
    _close(m1, x1[:, 0], 0, 0, "H=1 mean")

    a, b = 1.5, -0.25
    d = (a - b) / 2
    y2 = O.layer_norm_forward(np.array([[a, b]]), None, None, eps)[0]
    k = d / np.sqrt(d * d + eps)
    _close(y2, [[k, -k]], 1e-14, 0, "two-element row")

    c = np.array([[0.5, 0.5, 0.5, 0.5]])
    g4 = np.array([1.0, 2.0, -3.0, 0.1])
    yr = O.rms_norm_forward(c, g4, eps)[0]
    _close(yr, [g4 * 0.5 / np.sqrt(0.25 + eps)], 1e-14, 0, "rms const row")

    r = _rng(7)
    xs = 10 + 0.5 * r.standard_normal((4, 50))
    z = (xs - xs.mean(axis=1, keepdims=True)) / np.sqrt(xs.var(axis=1, keepdims=True) + eps)
    _close(O.layer_norm_forward(xs, None, None, eps)[0], z, 1e-12, 1e-12, "standard score")


# --------------------------------------------------------------------------
# statistics: Welford and the parallel merge
# --------------------------------------------------------------------------

def pin_welford(O):
    r = _rng(11)
    for H, off in [(1, 0.0), (7, 0.0), (64, 1000.0), (1000, -3.0), (2049, 1e4)]:
        v = off + 0.01 * r.standard_normal(H)
        n, mean, m2 = O.welford_sequential(v)
        assert n == H
        _close(mean, np.mean(v), 1e-13, 0, "welford mean vs numpy")
        _close(m2 / H, np.var(v), 1e-9, 1e-18, "welford var vs numpy")
        tm, tv = O.two_pass_stats(v[None, :])
        _close(mean, tm[0], 1e-13, 0, "welford vs two-pass mean")
        _close(m2 / H, tv[0], 1e-9, 1e-18, "welford vs two-pass var")
        for trial in range(4):
            cuts = r.integers(0, H + 1, size=r.integers(0, 9))
            tn, tmean, tm2 = O.welford_tree(v, cuts)
            assert tn == H
            _close(tmean, np.mean(v), 1e-13, 0, "merge-tree mean")
            _close(tm2 / H, np.var(v), 1e-9, 1e-18, "merge-tree var")
    # the identity element and a two-chunk merge checked by hand
    assert O.welford_merge((0.0, 0.0, 0.0), (0.0, 0.0, 0.0)) == (0.0, 0.0, 0.0)
    n, m, m2 = O.welford_merge((2.0, 1.0, 2.0), (2.0, 5.0, 2.0))   # {0,2} and {4,6}
    assert (n, m, m2) == (4.0, 3.0, 20.0)


# --------------------------------------------------------------------------
# fused add
# --------------------------------------------------------------------------

def pin_fused(O):
    """h is the exact sum rounded as the page stores it; y is RMSNorm of h.

    bf16 + bf16 in fp32 is exact when the exponents differ by at most 16, so
    for such inputs the stored bf16 h equals torch's own bf16 cast of the
    exact sum.  y must equal torch's rms_norm of the exact sum.
    """
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-6
        x, gamma, _, _, res = _case(100 + i, N, H)
        xb = torch.from_numpy(x).to(torch.bfloat16).double()
        rb = torch.from_numpy(res).to(torch.bfloat16).double()
        y, h_st, rstd = O.fused_add_rms_norm_forward(xb.numpy(), rb.numpy(), gamma, eps, "bfloat16")
        exact = (xb + rb)
        _close(h_st, exact.to(torch.bfloat16).double().numpy(), 0, 0, "fused h")
        yt = F.rms_norm(exact, (H,), torch.from_numpy(gamma), eps).numpy()
        _close(y, yt, 1e-12, 1e-12, "fused y")
        _close(rstd, 1.0 / np.sqrt((exact.numpy() ** 2).mean(axis=1) + eps), 1e-12, 0, "fused rstd")


def pin_fused_backward_from_h(O):
    """The stored-h form of the fused backward.

    * With h = x + res exactly, it equals the (x, res) form (which finite
      differences pin) for both inputs' gradient and dgamma.
    * The residual-stream gradient enters linearly: the result minus
      dh_stream is independent of dh_stream, and equals torch autograd of
      rms_norm(h) plus dh_stream.
    """
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-6
        x, gamma, _, dy, res = _case(110 + i, N, H)
        h = x + res
        dx, dres, dg = O.fused_add_rms_norm_backward(dy, x, res, gamma, eps)
        dh, dg2 = O.fused_add_rms_norm_backward_from_h(dy, h, gamma, eps)
        _close(dh, dx, 1e-13, 1e-13, "from-h dh vs dx")
        _close(dh, dres, 1e-13, 1e-13, "from-h dh vs dres")
        _close(dg2, dg, 1e-13, 1e-13, "from-h dgamma")
        stream = _rng(120 + i).standard_normal((N, H))
        dh_s, dg_s = O.fused_add_rms_norm_backward_from_h(dy, h, gamma, eps, stream)
        tdx, tdg, _ = _autograd(lambda a, g, b: F.rms_norm(a, (H,), g, eps), h, gamma, None, dy)
        _close(dh_s, tdx + stream, 1e-9, 1e-11, "from-h with stream vs autograd")
        _close(dg_s, tdg, 1e-9, 1e-11, "from-h dgamma vs autograd")


def pin_backward_from_output(O):
    """The saved-output form of the backward.

    * Fed the exact forward output and rstd, it equals the x form (pinned
      above by autograd and finite differences), with and without gamma/beta.
    * It is a function of (dy, y, rstd, gamma, beta) alone: a row rescaled in
      rstd scales dx by the same factor and leaves dgamma, dbeta unchanged.
    """
    for i, (N, H) in enumerate(SHAPES):
        eps = 1e-5
        x, gamma, beta, dy, _ = _case(130 + i, N, H)
        for g, b in ((gamma, beta), (None, None), (gamma, None)):
            y, _, rstd = O.layer_norm_forward(x, g, b, eps)
            want = O.layer_norm_backward(dy, x, g, eps)
            got = O.layer_norm_backward_from_output(dy, y, rstd, g, b)
            for a_, w_, nm in zip(got, want, ("dx", "dgamma", "dbeta")):
                _close(a_, w_, 1e-10, 1e-12, f"LN from-output {nm}")
            yr, rr = O.rms_norm_forward(x, g, eps)
            want = O.rms_norm_backward(dy, x, g, eps)
            got = O.rms_norm_backward_from_output(dy, yr, rr, g)
            for a_, w_, nm in zip(got, want, ("dx", "dgamma")):
                _close(a_, w_, 1e-10, 1e-12, f"RMS from-output {nm}")
        y, _, rstd = O.layer_norm_forward(x, gamma, beta, eps)
        k = np.linspace(0.5, 2.0, N)
        a1 = O.layer_norm_backward_from_output(dy, y, rstd, gamma, beta)
        a2 = O.layer_norm_backward_from_output(dy, y, rstd * k, gamma, beta)
        _close(a2[0], a1[0] * k[:, None], 1e-12, 1e-12, "dx linear in rstd")
        _close(a2[1], a1[1], 0, 0, "dgamma independent of rstd")


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------

def pin_bf16_rounding(O):
    r = _rng(5)
    vals = np.concatenate([
        r.standard_normal(20000) * 10.0 ** r.integers(-30, 30, 20000),
        # exact ties: 1 + k*2^-8 sits halfway between bfloat16 neighbours for odd k
        1.0 + np.arange(1, 64, 2) * 2.0 ** -8,
        -(1.0 + np.arange(1, 64, 2) * 2.0 ** -8),
        [0.0, -0.0, 3.3895313892515355e38, 3.4e38, 1e-40, -1e-42, np.inf, -np.inf],
    ])
    f32 = vals.astype(np.float32)
    mine = O.round_to_bfloat16(f32)
    ref = torch.from_numpy(f32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(mine, ref), "bf16 rounding differs from torch"
    assert np.all(np.isnan(O.round_to_bfloat16(np.array([np.nan], dtype=np.float32))))
    _close(O.round_to_float32(np.array([1.0 + 2.0 ** -30])), [1.0], 0, 0, "f32 rounding")


def pin_f16_rounding(O):
    r = _rng(6)
    vals = np.concatenate([
        r.standard_normal(20000) * 10.0 ** r.integers(-9, 6, 20000),
        # exact ties: 1 + k*2^-11 sits halfway between binary16 neighbours for odd k
        1.0 + np.arange(1, 64, 2) * 2.0 ** -11,
        -(1.0 + np.arange(1, 64, 2) * 2.0 ** -11),
        # subnormal ties (k*2^-25, k odd) and the overflow threshold
        np.arange(1, 40, 2) * 2.0 ** -25,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -26, np.inf, -np.inf],
    ])
    f32 = vals.astype(np.float32)
    mine = O.round_to_float16(f32)
    ref = torch.from_numpy(f32).to(torch.float16).double().numpy()
    assert np.array_equal(mine, ref), "fp16 rounding differs from torch"
    assert O.round_to_float16(np.array([65519.0]))[0] == 65504.0
    assert np.isinf(O.round_to_float16(np.array([65520.0]))[0])
    assert O.round_to_float16(np.array([3 * 2.0 ** -25]))[0] == 2.0 ** -23  # tie to even (2 units)
    assert np.all(np.isnan(O.round_to_float16(np.array([np.nan], dtype=np.float32))))


ALL_PINS = [
    pin_ln_forward_vs_torch,
    pin_rms_forward_vs_torch,
    pin_ln_backward_vs_autograd,
    pin_rms_backward_vs_autograd,
    pin_fd_layer_norm,
    pin_fd_rms_norm,
    pin_fd_fused,
    pin_ln_invariants,
    pin_rms_invariants,
    pin_closed_forms,
    pin_welford,
    pin_fused,
    pin_fused_backward_from_h,
    pin_bf16_rounding,
    pin_f16_rounding,
    pin_backward_from_output,
]
