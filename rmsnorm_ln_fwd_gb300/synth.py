"""Seeded synthetic inputs for row-wise LayerNorm / RMSNorm workloads.

This module only draws random numbers; it holds none of the normalisation
arithmetic.  Tests, the benchmark and the smoke check feed the same tensors
to the CUDA library and to the CPU oracle.

Recipe (every tensor drawn in fp32 on the CPU from its own seeded
``torch.Generator``, then cast once to its storage dtype):

* x, residual, dy, dh_stream ~ N(0, 1)  (x = offset + scale * N(0, 1) for the
  large-offset stability workload, e.g. offset 1000, scale 1e-2);
* gamma = 1 + 0.1 * N(0, 1);  beta = 0.1 * N(0, 1).
"""

from __future__ import annotations

import torch

# One independent generator stream per tensor role, so a tensor's values do
# not depend on which other tensors are drawn or on their shapes.
_STREAM = {"x": 1, "gamma": 2, "beta": 3, "dy": 4, "residual": 5, "dh_stream": 6}

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _gen(seed: int, role: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + _STREAM[role])
    return g


def normal(shape, seed: int, role: str, *, mean: float = 0.0, std: float = 1.0,
           dtype=torch.float32) -> torch.Tensor:
    """mean + std * N(0, 1), drawn in fp32 on the CPU, then cast to ``dtype``."""
    z = torch.randn(tuple(shape), generator=_gen(seed, role), dtype=torch.float32)
    if std != 1.0:
        z.mul_(std)
    if mean != 0.0:
        z.add_(mean)
    return z.to(dtype)


def norm_inputs(N: int, H: int, dtype="bf16", w_dtype=None, seed: int = 0, *,
                x_offset: float = 0.0, x_scale: float = 1.0,
                with_beta: bool = True, with_dy: bool = True,
                with_residual: bool = False, with_dh_stream: bool = False) -> dict:
    """CPU tensors for one (N, H) workload: x, gamma, beta, dy, residual and
    dh_stream (a gradient arriving through the stored residual sum)."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    wdt = dt if w_dtype is None else (DTYPES[w_dtype] if isinstance(w_dtype, str) else w_dtype)
    out = {
        "x": normal((N, H), seed, "x", mean=x_offset, std=x_scale, dtype=dt),
        "gamma": normal((H,), seed, "gamma", mean=1.0, std=0.1, dtype=wdt),
    }
    if with_beta:
        out["beta"] = normal((H,), seed, "beta", std=0.1, dtype=wdt)
    if with_dy:
        out["dy"] = normal((N, H), seed, "dy", dtype=dt)
    if with_residual:
        out["residual"] = normal((N, H), seed, "residual", dtype=dt)
    if with_dh_stream:
        out["dh_stream"] = normal((N, H), seed, "dh_stream", dtype=dt)
    return out
