"""The wide-chunk forward kernel at its boundaries, against the fp64 oracle.

Half-precision LayerNorm and RMSNorm rows of at least 512 columns (a multiple
of 16) whose rows are 32-byte aligned take 32-byte chunks of 16 contiguous
columns a thread.  The cases straddle its shapes: one chunk a lane (512),
a second chunk on some lanes only (528, 768, 1040), one warp a row at two
chunks (1024), several warps (5120, 8192, 16384), the 640-thread limit (20480)
and the first width past it (20496, which takes the cluster rows).  They run
tiny and ragged row counts, padded strides that keep 32-byte alignment and
ones that keep only 16-byte alignment (the 16-byte register rows), fp32
parameters, missing gamma/beta, and rows whose shift sits far from the mean
(the exact second pass).  The fused add takes one chunk a thread: its widths,
h written over x or the residual, and padded strides, h checked bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import DT_NAME, DT_ORACLE, check_mean, check_out, check_rstd, ln_y_scale, np64, rms_y_scale
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF, F16, F32 = torch.bfloat16, torch.float16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _strided(src, ld):
    N, H = src.shape
    buf = torch.zeros(N * ld + 64, dtype=src.dtype, device=src.device)
    v = buf[:N * ld].view(N, ld)[:, :H]
    v.copy_(src)
    return v


def _run(kind, N, H, dt, ld=None, wdt=None, affine=True, far_pivot=False, seed=5):
    eps = 1e-5
    t = {k: v.to(DEV) for k, v in synth.norm_inputs(N, H, DT_NAME[dt], None if wdt is None else DT_NAME[wdt],
                                                     seed).items()}
    x = t["x"]
    if far_pivot:  # column 0 an outlier on some rows, the rest of the row offset on others
        x = x.clone()
        x[0::3, 0] = 40.0
        x[1::3, 1:] += 25.0
    xs = _strided(x, ld) if ld is not None else x
    yb = _strided(torch.zeros_like(x), ld) if ld is not None else None
    g = t["gamma"] if affine else None
    xn = np64(x)
    gn = None if g is None else np64(g)
    what = f"{kind} {N}x{H} ld={ld}"
    if kind == "ln":
        b = t["beta"] if affine else None
        bn = None if b is None else np64(b)
        y, mean, rstd = nl.ln_forward(xs, g, b, eps, out=yb)
        torch.cuda.synchronize()
        yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
        check_out(np64(y), yr, ln_y_scale(xn, mr, rr, gn, bn), dt, what + " y")
        check_mean(np64(mean), mr, xn, what + " mean")
    else:
        y, rstd = nl.rms_forward(xs, g, eps, out=yb)
        torch.cuda.synchronize()
        yr, rr = O.rms_norm_forward(xn, gn, eps)
        check_out(np64(y), yr, rms_y_scale(xn, rr, gn), dt, what + " y")
    check_rstd(np64(rstd), rr, what + " rstd")
    if ld is not None and ld > H:  # the padding between rows stays untouched
        pad = yb.as_strided((N - 1, ld - H), (ld, 1), yb.storage_offset() + H)
        assert torch.count_nonzero(pad) == 0, "y padding written"


@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [512, 528, 768, 1024, 1040, 2048, 5120, 8192, 16384, 20480, 20496])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_wide_widths(kind, H, dt):
    _run(kind, 300, H, dt)


@pytest.mark.parametrize("N", [1, 7, 151, 305, 2049])
@pytest.mark.parametrize("H", [1024, 5120, 16384])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_wide_row_counts(kind, N, H):
    _run(kind, N, H, BF, seed=N)


@pytest.mark.parametrize("H,ld", [(1024, 1040), (1024, 1032), (5120, 5136), (5120, 5128), (528, 544), (16384, 16400)])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_wide_strides(kind, H, ld):
    # ld - H = 16 elements keeps every row 32-byte aligned (wide chunks); 8
    # keeps 16-byte alignment only (16-byte register rows)
    _run(kind, 97, H, BF, ld=ld)


@pytest.mark.parametrize("H", [1024, 5120])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_wide_fp32_params_and_no_affine(kind, H):
    _run(kind, 200, H, BF, wdt=F32)
    _run(kind, 200, H, F16, affine=False)


@pytest.mark.parametrize("H", [528, 1024, 5120, 16384])
@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
def test_wide_pivot_far_from_mean(H, dt):
    _run("ln", 48, H, dt, far_pivot=True)


def _fused(N, H, dt, inplace=None, ld=None, seed=11):
    eps = 1e-6
    t = {k: v.to(DEV) for k, v in synth.norm_inputs(N, H, DT_NAME[dt], seed=seed, with_beta=False, with_dy=False,
                                                     with_residual=True).items()}
    x0, r0 = t["x"].clone(), t["residual"].clone()
    x, r = (_strided(t["x"], ld), _strided(t["residual"], ld)) if ld is not None else (t["x"], t["residual"])
    h_out = {"x": x, "residual": r, None: None}[inplace]
    if ld is not None and inplace is None:
        h_out = _strided(torch.zeros_like(x0), ld)
    y, h, rstd = nl.fused_add_rms_forward(x, r, t["gamma"], eps, h_out=h_out)
    torch.cuda.synchronize()
    xn, rn, gn = np64(x0), np64(r0), np64(t["gamma"])
    yr, hr, rr = O.fused_add_rms_norm_forward(xn, rn, gn, eps, DT_ORACLE[dt])
    assert np.array_equal(np64(h), hr), f"fused h {N}x{H} ld={ld} inplace={inplace}: not bit-exact"
    check_out(np64(y), yr, rms_y_scale(xn + rn, rr, gn), dt, f"fused y {N}x{H}")
    check_rstd(np64(rstd), rr, f"fused rstd {N}x{H}")


@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [512, 528, 1040, 5120, 10240, 10256])
def test_wide_fused_widths(H, dt):
    _fused(300, H, dt)


@pytest.mark.parametrize("inplace", ["x", "residual"])
@pytest.mark.parametrize("H", [1024, 5120])
def test_wide_fused_in_place(H, inplace):
    _fused(257, H, BF, inplace=inplace)


@pytest.mark.parametrize("H,ld", [(1024, 1040), (1024, 1032), (5120, 5136)])
def test_wide_fused_strides(H, ld):
    _fused(97, H, BF, ld=ld)
