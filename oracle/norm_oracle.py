"""Plain fp64 CPU oracle for row-wise LayerNorm and RMSNorm.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
table or helper with the CUDA library.

Every function takes numpy arrays holding the exact values the GPU sees
(inputs already rounded to their storage dtype) and computes in float64 with
whole-array numpy operations, one formula per line, in the order the pages
state them.  There is no blocking, fusion or reordering beyond that.

Sources (page title -- section):

* "Skill: Write a Triton LayerNorm Kernel" -- Required reasoning process,
  steps 3-10; Kernel design rules; Correctness requirements.
* "Skill: Write CUDA LayerNorm Kernel" -- Required reasoning process,
  steps 2 (Welford recurrence), 3 (parallel merge), 5-8 (normalise, affine,
  epsilon, backward formulas).
* "Skill: Write a Triton Fused Add+RMSNorm Kernel" -- Required reasoning
  process, steps 3-7 and 10.
* The RMSNorm backward is not printed on any page; ``rms_norm_backward``
  derives it from the RMSNorm forward (derivation in its docstring).

Pinning: every function here is pinned by ``tests/test_oracle.py`` against
finite differences, invariants of the mathematics, closed forms, torch's CPU
fp64 library routines and brute force on tiny inputs.  No function is
"parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "layer_norm_forward",
    "rms_norm_forward",
    "fused_add_rms_norm_forward",
    "layer_norm_backward",
    "rms_norm_backward",
    "layer_norm_backward_from_output",
    "rms_norm_backward_from_output",
    "fused_add_rms_norm_backward",
    "fused_add_rms_norm_backward_from_h",
    "welford_sequential",
    "welford_merge",
    "welford_tree",
    "two_pass_stats",
    "round_to_float32",
    "round_to_bfloat16",
    "round_to_float16",
    "round_to_dtype",
]


def _f64_2d(a):
    a = np.asarray(a, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("expected a 2-D (rows, H) array")
    return a


def _param(p, H, fill):
    if p is None:
        return np.full(H, fill, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    if p.shape != (H,):
        raise ValueError("a parameter must have shape (H,)")
    return p


# ---------------------------------------------------------------------------
# Statistics.  Two-pass (mean first, then the sum of squared deviations) is the
# definition; Welford's recurrence and the parallel merge reach the same
# numbers and are kept here so the pin tests can compare the two.
# ---------------------------------------------------------------------------

def two_pass_stats(x):
    """Per-row (mean, biased variance) by the two-pass definition.

    "Skill: Write a Triton LayerNorm Kernel", Required reasoning process,
    steps 3 and 5: mean = sum(x)/H, var = sum((x - mean)^2)/H -- the divisor
    is the full row length H.
    """
    x = _f64_2d(x)
    H = x.shape[1]
    mean = x.sum(axis=1) / H
    centred = x - mean[:, None]
    var = (centred * centred).sum(axis=1) / H
    return mean, var


def welford_sequential(values):
    """Welford's online recurrence over a 1-D sequence -> (count, mean, M2).

    "Skill: Write CUDA LayerNorm Kernel", Required reasoning process, step 2:
    mean_new = mean_old + (x - mean_old)/n and
    M2_new = M2_old + (x - mean_old)(x - mean_new); var = M2 / count.
    Pure-Python loop: for small inputs only.
    """
    count, mean, m2 = 0.0, 0.0, 0.0
    for v in np.asarray(values, dtype=np.float64).ravel():
        count += 1.0
        old = mean
        mean = old + (v - old) / count
        m2 = m2 + (v - old) * (v - mean)
    return count, mean, m2


def welford_merge(a, b):
    """Parallel Welford merge of two (count, mean, M2) triples.

    "Skill: Write CUDA LayerNorm Kernel", Required reasoning process, step 3:
    n = n_a + n_b; delta = mean_b - mean_a; mean = mean_a + delta*n_b/n;
    M2 = M2_a + M2_b + delta^2 * n_a * n_b / n.  A triple with count 0 is the
    identity (step 4).
    """
    na, ma, m2a = a
    nb, mb, m2b = b
    n = na + nb
    if n == 0:
        return 0.0, 0.0, 0.0
    delta = mb - ma
    mean = ma + delta * nb / n
    m2 = m2a + m2b + delta * delta * na * nb / n
    return n, mean, m2


def welford_tree(values, split_points):
    """Welford over the chunks cut at ``split_points``, merged left to right.

    Models the per-thread accumulators of a parallel reduction followed by the
    merge of step 3 on the CUDA page.  Empty chunks contribute the identity.
    """
    values = np.asarray(values, dtype=np.float64).ravel()
    bounds = [0] + sorted(int(s) for s in split_points) + [values.size]
    acc = (0.0, 0.0, 0.0)
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        acc = welford_merge(acc, welford_sequential(values[lo:hi]))
    return acc


# ---------------------------------------------------------------------------
# Forward passes.
# ---------------------------------------------------------------------------

def layer_norm_forward(x, gamma=None, beta=None, eps=1e-5):
    """LayerNorm forward over the last dim -> (y, mean, rstd), all float64.

    "Skill: Write a Triton LayerNorm Kernel", Required reasoning process,
    steps 3-10: mean = sum(x)/H; var = sum((x-mean)^2)/H;
    rstd = 1/sqrt(var + eps) (eps inside the square root);
    x_hat = (x - mean)*rstd; y = x_hat*gamma + beta.  gamma/beta of shape
    (H,) are indexed by column only; ``None`` means the identity (1 and 0).
    mean and rstd are the per-row values saved for the backward.
    """
    x = _f64_2d(x)
    H = x.shape[1]
    if not eps > 0:
        raise ValueError("eps must be strictly positive")
    g = _param(gamma, H, 1.0)
    b = _param(beta, H, 0.0)
    mean, var = two_pass_stats(x)
    rstd = 1.0 / np.sqrt(var + eps)
    x_hat = (x - mean[:, None]) * rstd[:, None]
    y = x_hat * g[None, :] + b[None, :]
    return y, mean, rstd


def rms_norm_forward(x, gamma=None, eps=1e-5):
    """RMSNorm forward -> (y, rstd), float64.

    "Skill: Write a Triton LayerNorm Kernel", step 5 (RMSNorm branch) and
    "Skill: Write CUDA LayerNorm Kernel", Kernel design rules (RMSNorm):
    mean_sq = sum(x^2)/H; rstd = 1/sqrt(mean_sq + eps); y = x*rstd*gamma.
    No mean subtraction and no beta.
    """
    x = _f64_2d(x)
    H = x.shape[1]
    if not eps > 0:
        raise ValueError("eps must be strictly positive")
    g = _param(gamma, H, 1.0)
    mean_sq = (x * x).sum(axis=1) / H
    rstd = 1.0 / np.sqrt(mean_sq + eps)
    y = x * rstd[:, None] * g[None, :]
    return y, rstd


def fused_add_rms_norm_forward(x, residual, gamma=None, eps=1e-6, h_dtype="float32"):
    """Fused residual add + RMSNorm forward -> (y, h_stored, rstd).

    "Skill: Write a Triton Fused Add+RMSNorm Kernel", Required reasoning
    process, steps 3-7:
      * h = x + residual, formed in fp32 (step 3).  The summed residual that
        the kernel writes back is that fp32 sum cast to the input dtype
        (step 4), so ``h_stored`` = round_to_dtype(round_to_float32(x + res)).
        Both roundings are the page's own, so the stored integer bit pattern
        is decided in the page's precision.
      * mean_sq = sum(h^2)/H; rstd = 1/sqrt(mean_sq + eps) (step 5);
        y = h*rstd*gamma (step 6), computed here from the exact (float64)
        sum -- the page keeps h in fp32 registers, never the rounded copy.
    """
    x = _f64_2d(x)
    r = _f64_2d(residual)
    if x.shape != r.shape:
        raise ValueError("x and residual must have the same shape")
    h = x + r
    h_stored = round_to_dtype(round_to_float32(h), h_dtype)
    y, rstd = rms_norm_forward(h, gamma, eps)
    return y, h_stored, rstd


# ---------------------------------------------------------------------------
# Backward passes.  The oracle recomputes the statistics in float64 from x;
# the GPU path reads the saved fp32 mean/rstd instead.
# ---------------------------------------------------------------------------

def layer_norm_backward(dy, x, gamma=None, eps=1e-5):
    """LayerNorm backward -> (dx, dgamma, dbeta), float64.

    "Skill: Write CUDA LayerNorm Kernel", Required reasoning process, step 8:
      dgamma_j = sum over all rows of x_hat_j * dy_j
      dbeta_j  = sum over all rows of dy_j
      dx_j = (1/H) * rstd * (H*g_j - sum(g) - x_hat_j * sum(g * x_hat)),
    where g_j = dy_j * gamma_j is the gradient reaching x_hat (the page's
    "dL/dy_hat").  The parameter sums run over every row, i.e. over the batch
    and sequence dims together (Common failure modes, last bullet).
    """
    dy = _f64_2d(dy)
    x = _f64_2d(x)
    if dy.shape != x.shape:
        raise ValueError("dy and x must have the same shape")
    H = x.shape[1]
    gm = _param(gamma, H, 1.0)
    mean, var = two_pass_stats(x)
    rstd = 1.0 / np.sqrt(var + eps)
    x_hat = (x - mean[:, None]) * rstd[:, None]
    g = dy * gm[None, :]
    sum_g = g.sum(axis=1)
    sum_g_xhat = (g * x_hat).sum(axis=1)
    dx = (rstd[:, None] / H) * (H * g - sum_g[:, None] - x_hat * sum_g_xhat[:, None])
    dgamma = (dy * x_hat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    return dx, dgamma, dbeta


def rms_norm_backward(dy, x, gamma=None, eps=1e-5):
    """RMSNorm backward -> (dx, dgamma), float64.

    No page prints this formula; it is derived from the RMSNorm forward
    y_j = gamma_j * x_j * r with r = (m + eps)^(-1/2), m = sum(x^2)/H:
      dr/dx_k = -r^3 x_k / H, so with g_j = dy_j*gamma_j and x_hat = x*r,
      dx_k = r * (g_k - x_hat_k * sum_j(g_j * x_hat_j) / H),
      dgamma_j = sum over all rows of dy_j * x_hat_j.
    """
    dy = _f64_2d(dy)
    x = _f64_2d(x)
    if dy.shape != x.shape:
        raise ValueError("dy and x must have the same shape")
    H = x.shape[1]
    gm = _param(gamma, H, 1.0)
    mean_sq = (x * x).sum(axis=1) / H
    rstd = 1.0 / np.sqrt(mean_sq + eps)
    x_hat = x * rstd[:, None]
    g = dy * gm[None, :]
    c2 = (g * x_hat).sum(axis=1) / H
    dx = rstd[:, None] * (g - x_hat * c2[:, None])
    dgamma = (dy * x_hat).sum(axis=0)
    return dx, dgamma


def layer_norm_backward_from_output(dy, y, rstd, gamma=None, beta=None):
    """LayerNorm backward from the saved output -> (dx, dgamma, dbeta), float64.

    The step 8 formulas of "Skill: Write CUDA LayerNorm Kernel" (as in
    ``layer_norm_backward``), with x_hat recovered from the forward's output
    instead of recomputed from x: y = x_hat*gamma + beta gives
    x_hat = (y - beta) / gamma.  "Rewrite Triton normalization backward
    kernel_1 (#499)", Benchmark harness, has the backward read the forward's
    saved output.  ``rstd`` is the forward's saved 1/sqrt(var + eps) per row
    (it cannot be recovered from y).  Columns with gamma = 0 carry no
    information about x_hat and give non-finite results there.
    """
    dy = _f64_2d(dy)
    y = _f64_2d(y)
    if dy.shape != y.shape:
        raise ValueError("dy and y must have the same shape")
    H = y.shape[1]
    gm = _param(gamma, H, 1.0)
    bt = _param(beta, H, 0.0)
    rstd = np.asarray(rstd, dtype=np.float64).reshape(-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        x_hat = (y - bt[None, :]) / gm[None, :]
    g = dy * gm[None, :]
    sum_g = g.sum(axis=1)
    sum_g_xhat = (g * x_hat).sum(axis=1)
    dx = (rstd[:, None] / H) * (H * g - sum_g[:, None] - x_hat * sum_g_xhat[:, None])
    dgamma = (dy * x_hat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    return dx, dgamma, dbeta


def rms_norm_backward_from_output(dy, y, rstd, gamma=None):
    """RMSNorm backward from the saved output -> (dx, dgamma), float64.

    The ``rms_norm_backward`` formulas with x_hat = y / gamma recovered from
    the forward's output y = x_hat*gamma; ``rstd`` is the forward's saved
    1/sqrt(mean(x^2) + eps).
    """
    dy = _f64_2d(dy)
    y = _f64_2d(y)
    if dy.shape != y.shape:
        raise ValueError("dy and y must have the same shape")
    H = y.shape[1]
    gm = _param(gamma, H, 1.0)
    rstd = np.asarray(rstd, dtype=np.float64).reshape(-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        x_hat = y / gm[None, :]
    g = dy * gm[None, :]
    c2 = (g * x_hat).sum(axis=1) / H
    dx = rstd[:, None] * (g - x_hat * c2[:, None])
    dgamma = (dy * x_hat).sum(axis=0)
    return dx, dgamma


def fused_add_rms_norm_backward(dy, x, residual, gamma=None, eps=1e-6):
    """Backward of y = rmsnorm(x + residual)*gamma -> (dx, dresidual, dgamma).

    "Skill: Write a Triton Fused Add+RMSNorm Kernel", Required reasoning
    process, step 10: dh/dx = dh/dres = 1, so both inputs receive the RMSNorm
    gradient with respect to h, unchanged.  Gradients arriving through the
    stored h (the residual stream) are not part of this function.
    """
    h = _f64_2d(x) + _f64_2d(residual)
    dh, dgamma = rms_norm_backward(dy, h, gamma, eps)
    return dh, dh.copy(), dgamma


def fused_add_rms_norm_backward_from_h(dy, h, gamma=None, eps=1e-6, dh_stream=None):
    """Backward of the fused add from the stored h -> (dh, dgamma).

    "Skill: Write a Triton Fused Add+RMSNorm Kernel", Required reasoning
    process steps 9-10: training keeps rstd and the summed activation h (the
    stored copy is what the backward can read); the RMSNorm gradient with
    respect to h is formed once and is the gradient of both x and residual
    (dh/dx = dh/dres = 1).  ``dh_stream`` is the gradient arriving through
    the stored h itself (the residual stream's consumers), added to that same
    total: dL/dh = rmsnorm_backward(dy, h) + dh_stream.
    """
    dh, dgamma = rms_norm_backward(dy, h, gamma, eps)
    if dh_stream is not None:
        dh = dh + _f64_2d(dh_stream)
    return dh, dgamma


# ---------------------------------------------------------------------------
# Storage rounding (round to nearest, ties to even), written out on the bits.
# ---------------------------------------------------------------------------

def round_to_float32(a):
    """float64 -> nearest float32 (ties to even), returned as float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to_bfloat16(a):
    """float32-representable values -> nearest bfloat16 (ties to even), as float64.

    bfloat16 keeps the top 16 bits of a float32.  Round to nearest even on
    the dropped 16 bits: add 0x7FFF plus the lowest kept bit, then truncate.
    NaN stays NaN; values that round past the largest finite bfloat16 become
    infinity, as IEEE rounding prescribes.
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) << np.uint64(16)
    out = (rounded & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(f)
    if np.any(nan):
        out = np.where(nan, np.nan, out)
    return out


def round_to_float16(a):
    """float32-representable values -> nearest IEEE binary16 (ties to even), as float64.

    numpy's float32 -> float16 conversion is the rounding step: binary16 keeps
    10 fraction bits, has subnormals down to 2^-24, and values from 65520 up
    round to infinity.
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    with np.errstate(over="ignore"):
        return f.astype(np.float16).astype(np.float64)


def round_to_dtype(a, dtype):
    """Round float64 values to the storage dtype named by ``dtype``."""
    name = str(dtype).replace("torch.", "")
    if name in ("float32", "f32", "fp32"):
        return round_to_float32(a)
    if name in ("bfloat16", "bf16"):
        return round_to_bfloat16(a)
    if name in ("float16", "f16", "fp16", "half"):
        return round_to_float16(a)
    if name in ("float64", "f64"):
        return np.asarray(a, dtype=np.float64)
    raise ValueError(f"unsupported dtype {dtype!r}")
