"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Sizes run from tiny to several tiles with ragged tails (small H sweep, N
sweep), plus the edge cases: H = 1, zero-variance rows, unaligned pointers and
strides (scalar path), padded row strides, in-place calls, fp32 parameters
with bf16 rows, missing gamma/beta, N = 0 and guard bands around every output.
The backward is fed the GPU forward's saved mean/rstd, as in training.
"""

import numpy as np
import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import (DT_NAME, DT_ORACLE, Guarded, check_bf16, check_f32, check_mean, check_out, check_param,
                      check_rstd, ln_dx_scale, ln_y_scale, np64, rms_dx_scale, rms_y_scale)
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF, F32, F16 = torch.bfloat16, torch.float32, torch.float16
DTS, DT_IDS = [BF, F32, F16], ["bf16", "f32", "f16"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _inputs(N, H, dt, seed=0, wdt=None, **kw):
    d = synth.norm_inputs(N, H, DT_NAME[dt], None if wdt is None else DT_NAME[wdt], seed, **kw)
    return {k: v.to(DEV) for k, v in d.items()}


def ln_case(N, H, dt, eps=1e-5, seed=0, wdt=None, gamma=True, beta=True, **kw):
    t = _inputs(N, H, dt, seed, wdt, with_residual=False, **kw)
    g = t["gamma"] if gamma else None
    b = t["beta"] if beta else None
    y, mean, rstd = nl.ln_forward(t["x"], g, b, eps)
    dx, dg, db = nl.ln_backward(t["dy"], t["x"], mean, rstd, g)
    torch.cuda.synchronize()
    x, dy = np64(t["x"]), np64(t["dy"])
    gn = None if g is None else np64(g)
    bn = None if b is None else np64(b)
    yr, mr, rr = O.layer_norm_forward(x, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dy, x, gn, eps)
    check_out(np64(y), yr, ln_y_scale(x, mr, rr, gn, bn), dt, f"ln y {N}x{H}")
    check_mean(np64(mean), mr, x, f"ln mean {N}x{H}")
    check_rstd(np64(rstd), rr, f"ln rstd {N}x{H}")
    check_out(np64(dx), dxr, ln_dx_scale(dy, x, gn, eps), dt, f"ln dx {N}x{H}")
    wd = dg.dtype
    check_param(np64(dg), dgr, wd, f"ln dgamma {N}x{H}")
    check_param(np64(db), dbr, wd, f"ln dbeta {N}x{H}")


def rms_case(N, H, dt, eps=1e-5, seed=0, wdt=None, gamma=True, **kw):
    t = _inputs(N, H, dt, seed, wdt, with_beta=False, **kw)
    g = t["gamma"] if gamma else None
    y, rstd = nl.rms_forward(t["x"], g, eps)
    dx, dg = nl.rms_backward(t["dy"], t["x"], rstd, g)
    torch.cuda.synchronize()
    x, dy = np64(t["x"]), np64(t["dy"])
    gn = None if g is None else np64(g)
    yr, rr = O.rms_norm_forward(x, gn, eps)
    dxr, dgr = O.rms_norm_backward(dy, x, gn, eps)
    check_out(np64(y), yr, rms_y_scale(x, rr, gn), dt, f"rms y {N}x{H}")
    check_rstd(np64(rstd), rr, f"rms rstd {N}x{H}")
    check_out(np64(dx), dxr, rms_dx_scale(dy, x, gn, eps), dt, f"rms dx {N}x{H}")
    check_param(np64(dg), dgr, dg.dtype, f"rms dgamma {N}x{H}")


def fused_case(N, H, dt, eps=1e-6, seed=0, wdt=None, inplace=None):
    t = _inputs(N, H, dt, seed, wdt, with_beta=False, with_dy=False, with_residual=True)
    x0, r0 = t["x"].clone(), t["residual"].clone()
    h_out = {"x": t["x"], "residual": t["residual"], None: None}[inplace]
    y, h, rstd = nl.fused_add_rms_forward(t["x"], t["residual"], t["gamma"], eps, h_out=h_out)
    torch.cuda.synchronize()
    x, r, gn = np64(x0), np64(r0), np64(t["gamma"])
    yr, hr, rr = O.fused_add_rms_norm_forward(x, r, gn, eps, DT_ORACLE[dt])
    assert np.array_equal(np64(h), hr), f"fused h {N}x{H}: not bit-exact"
    check_out(np64(y), yr, rms_y_scale(x + r, rr, gn), dt, f"fused y {N}x{H}")
    check_rstd(np64(rstd), rr, f"fused rstd {N}x{H}")
    if inplace != "x":
        assert torch.equal(t["x"], x0), "x modified"
    if inplace != "residual":
        assert torch.equal(t["residual"], r0), "residual modified"


# ---------------------------------------------------------------------------
# the small LayerNorm configuration: (64, 256) fp32, every output checked
# ---------------------------------------------------------------------------

def test_ln_fp32_64x256():
    ln_case(64, 256, F32)


# ---------------------------------------------------------------------------
# H sweeps: warp-per-row, multi-warp rows, wide rows, loop path (H % VEC != 0
# or H beyond the register path), with ragged tails
# ---------------------------------------------------------------------------

H_SWEEP = [1, 2, 7, 8, 31, 32, 33, 64, 127, 128, 255, 256, 512, 768, 1000, 1024, 2048, 2049, 4095, 4096,
           5120, 8192, 16383, 16384, 20480, 32768, 40000]


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H", H_SWEEP)
def test_ln_sweep(H, dt):
    ln_case(37, H, dt, seed=H)


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H", H_SWEEP)
def test_rms_sweep(H, dt):
    rms_case(37, H, dt, seed=H + 1)


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H", H_SWEEP)
def test_fused_sweep(H, dt):
    fused_case(37, H, dt, seed=H + 2)


# P2's validation list: D in {64, 128, 512, 768, 1024, 2049}
@pytest.mark.parametrize("H", [64, 128, 512, 768, 1024, 2049])
@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
def test_ln_page_validation_widths(H, dt):
    ln_case(64, H, dt, seed=7 + H)


# ---------------------------------------------------------------------------
# N sweep: one row, fewer rows than SMs, an SM-count-plus-one, many rows (grid
# striding of the backward, several rows per partial)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 3, 153, 1000, 5000])
@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (256, F32), (2048, F32)], ids=["1024bf16", "5120bf16",
                                                                                         "256f32", "2048f32"])
def test_row_counts(N, H, dt):
    ln_case(N, H, dt, seed=N)
    rms_case(N, H, dt, seed=N + 1)


# ---------------------------------------------------------------------------
# two-CTA cluster rows of the backward (10240 < H <= 16384): row counts from
# one to beyond the resident cluster count, fp32 rows at 12288 columns, fp32
# parameters with half-precision rows (the parameter halves are offset by the
# parameter element size), and 16376 columns: in bf16 the halves are not whole
# 16-byte vectors (one CTA a row instead), in fp32 they are, with threads past
# the end of each half
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 3, 77, 500])
@pytest.mark.parametrize("H,dt", [(16384, BF), (16384, F16), (16384, F32), (12288, F32)],
                         ids=["16384bf16", "16384f16", "16384f32", "12288f32"])
def test_cluster_rows(N, H, dt):
    ln_case(N, H, dt, seed=N + H)
    rms_case(N, H, dt, seed=N + H + 1)


@pytest.mark.parametrize("N", [1, 5, 40])
@pytest.mark.parametrize("H,dt", [(24576, BF), (32768, BF), (65536, BF), (32768, F32)],
                         ids=["24576bf16", "32768bf16", "65536bf16", "32768f32"])
def test_cluster_rows_4_and_8(N, H, dt):
    """Rows past 16384 columns: clusters of four or eight CTAs a row."""
    ln_case(N, H, dt, seed=N + H)
    rms_case(N, H, dt, seed=N + H + 1)


@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
def test_cluster_rows_fp32_params(dt):
    ln_case(40, 16384, dt, wdt=F32, seed=9)
    rms_case(40, 16384, dt, wdt=F32, seed=10)


@pytest.mark.parametrize("H,dt", [(16376, BF), (16376, F32)], ids=["bf16", "f32"])
def test_wide_rows_without_whole_halves(H, dt):
    ln_case(37, H, dt, seed=11)
    rms_case(37, H, dt, seed=12)


# ---------------------------------------------------------------------------
# parameter variants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [1024, 5120, 1000])
def test_half_rows_fp32_params(H, dt):
    ln_case(64, H, dt, wdt=F32, seed=3)
    rms_case(64, H, dt, wdt=F32, seed=4)
    fused_case(64, H, dt, wdt=F32, seed=5)


@pytest.mark.parametrize("H", [256, 4096, 33])
@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
def test_no_affine(H, dt):
    ln_case(16, H, dt, gamma=False, beta=False, seed=11)
    ln_case(16, H, dt, gamma=True, beta=False, seed=12)
    rms_case(16, H, dt, gamma=False, seed=13)


# ---------------------------------------------------------------------------
# numerically special rows
# ---------------------------------------------------------------------------

def test_stability_offset_rows_fp32():
    """x = 1000 + 1e-2 N(0,1): the mean is 1e5 times the spread."""
    ln_case(8192, 1024, F32, x_offset=1000.0, x_scale=1e-2, seed=21)
    rms_case(8192, 1024, F32, x_offset=1000.0, x_scale=1e-2, seed=22)


@pytest.mark.parametrize("where", ["random", "fixed"])
@pytest.mark.parametrize("H", [1024, 5120, 16384])
@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
def test_ln_offset_outlier_rows(H, dt, where):
    """Rows constant at 1000 but for one outlier of a few storage spacings
    (|mean| * rstd above 1e3): the worst case for the saved fp32 mean's
    rounding inside x_hat.  Half an fp32 ulp of the mean shifts every x_hat by
    about 2e-4 here; through c2 = mean(g * x_hat) the shift reaches the
    outlier's dx multiplied by its x_hat (about 70), beyond one bf16 ulp at
    H = 5120 unless the backward removes it (the recentring).  dx elementwise
    and dgamma/dbeta in relative RMS must meet the stated bounds."""
    N, eps = 64, 1e-5
    t = _inputs(N, H, dt, seed=41)
    gen = torch.Generator().manual_seed(41)
    spacing = 4.0 if dt == BF else 0.5  # storage spacing at 1000
    x = torch.full((N, H), 1000.0)
    cols = torch.randint(0, H, (N,), generator=gen) if where == "random" else torch.full((N,), H // 3)
    k = torch.randint(1, 4, (N,), generator=gen).float()
    sign = torch.where(torch.rand(N, generator=gen) < 0.5, -1.0, 1.0)
    x[torch.arange(N), cols] = 1000.0 + 2.0 * spacing * k * sign
    x = x.to(dt)
    assert torch.equal(x.float()[torch.arange(N), cols], 1000.0 + 2.0 * spacing * k * sign), "values not exact"
    x = x.to(DEV)
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps)
    dx, dg, db = nl.ln_backward(t["dy"], x, mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    xn, gn, bn, dyn = np64(x), np64(t["gamma"]), np64(t["beta"]), np64(t["dy"])
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dyn, xn, gn, eps)
    assert np.all(np.abs(mr) * rr > 1e3), "rows are not offset enough to be a test"
    check_out(np64(y), yr, ln_y_scale(xn, mr, rr, gn, bn), dt, "outlier y")
    check_mean(np64(mean), mr, xn, "outlier mean")
    check_rstd(np64(rstd), rr, "outlier rstd")
    check_out(np64(dx), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, "outlier dx")
    check_param(np64(dg), dgr, dt, "outlier dgamma")
    check_param(np64(db), dbr, dt, "outlier dbeta")


@pytest.mark.parametrize("H", [1024, 5120, 1000])
def test_f16_small_activations(H):
    """|x| ~ 1e-3 in fp16: x*x would underflow in fp16; the statistics are fp32."""
    ln_case(64, H, F16, x_scale=1e-3, seed=61)
    rms_case(64, H, F16, x_scale=1e-3, seed=62)


@pytest.mark.parametrize("H", [1024, 1000])
def test_f16_output_overflow(H):
    """gamma = 40000 pushes |y| past 65504: those outputs round to +-inf,
    exactly where the oracle's rounding of the exact value does."""
    N, eps = 32, 1e-5
    t = _inputs(N, H, F16, seed=63)
    gamma = torch.full((H,), 40000.0, dtype=F16, device=DEV)
    y, _, _ = nl.ln_forward(t["x"], gamma, t["beta"], eps)
    yr_rms, _ = nl.rms_forward(t["x"], gamma, eps)
    torch.cuda.synchronize()
    x, bn = np64(t["x"]), np64(t["beta"])
    for got, (ref, *_) in ((np64(y), O.layer_norm_forward(x, np64(gamma), bn, eps)),
                           (np64(yr_rms), O.rms_norm_forward(x, np64(gamma), eps))):
        want = O.round_to_float16(ref)
        # away from the overflow threshold (65520) the inf pattern is decided
        sure = np.abs(np.abs(ref) - 65520.0) > 64.0
        assert np.any(np.isinf(want)), "case does not overflow"
        assert np.array_equal(np.isinf(got) & sure, np.isinf(want) & sure)
        assert np.array_equal(np.sign(got[np.isinf(got)]), np.sign(want[np.isinf(got)]))
        fin = np.isfinite(want) & sure
        err = np.abs(got[fin] - ref[fin])
        assert np.all(err <= 2.0 * np.abs(ref[fin]) * 2.0 ** -11 + 1e-3), "finite outputs"


@pytest.mark.parametrize("H", [64, 1024, 5120])
@pytest.mark.parametrize("dt", [BF, F32], ids=["bf16", "f32"])
def test_ln_pivot_far_from_mean(H, dt):
    """Rows whose first element (the kernels' shift) sits far from the mean:
    an outlier in column 0, or the whole row offset except column 0.  Both the
    one-reduction statistics and the exact second pass get exercised."""
    N, eps = 48, 1e-5
    t = _inputs(N, H, dt, seed=91)
    x = t["x"].clone()
    x[0::3, 0] = 40.0               # outlier pivot
    x[1::3, 1:] += 25.0             # pivot 25 below the rest of the row
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps)
    dx, dg, db = nl.ln_backward(t["dy"], x, mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    xn, gn, bn, dyn = np64(x), np64(t["gamma"]), np64(t["beta"]), np64(t["dy"])
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dyn, xn, gn, eps)
    # The kernels sum x - s for a shift s taken from the row's first 16-byte
    # vector; the fp32 rounding of the mean then scales with |s - mean| as
    # well as with the spread, so that distance joins the error scale of y.
    vec = 4 if dt == F32 else 8
    far = np.max(np.abs(xn[:, :vec] - mr[:, None]), axis=1)
    y_scale = ln_y_scale(xn, mr, rr, gn, bn) + (far * rr)[:, None] * np.abs(gn)[None, :]
    check_out(np64(y), yr, y_scale, dt, "pivot y")
    check_mean(np64(mean), mr, xn, "pivot mean")
    check_rstd(np64(rstd), rr, "pivot rstd")
    check_out(np64(dx), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, "pivot dx")
    check_param(np64(dg), dgr, dt, "pivot dgamma")
    check_param(np64(db), dbr, dt, "pivot dbeta")


@pytest.mark.parametrize("H", [1, 8, 1024, 5120, 40000])
@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
def test_zero_variance_rows(H, dt):
    """Constant rows: y = beta, rstd = eps^-1/2, dx = rstd*(g - mean(g))."""
    N, eps = 5, 1e-5
    t = _inputs(N, H, dt, seed=31)
    x = torch.full((N, H), 0.75, dtype=dt, device=DEV)
    x[1].fill_(-3.0)
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps)
    dx, dg, db = nl.ln_backward(t["dy"], x, mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    xn, gn, bn, dyn = np64(x), np64(t["gamma"]), np64(t["beta"]), np64(t["dy"])
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dyn, xn, gn, eps)
    assert np.array_equal(np64(y), np.broadcast_to(bn, (N, H)).astype(np.float64)), "y must equal beta exactly"
    check_mean(np64(mean), mr, xn, "mean")
    check_rstd(np64(rstd), rr, "rstd")
    check_out(np64(dx), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, "dx")
    check_param(np64(db), dbr, dt, "dbeta")
    assert np.max(np.abs(np64(dg))) <= 1e-6 * max(1.0, np.max(np.abs(dbr))), "dgamma must vanish"


# ---------------------------------------------------------------------------
# layouts: padded strides, misaligned pointers (scalar path), 3-D inputs
# ---------------------------------------------------------------------------

def _strided(src, ld, offset=0):
    N, H = src.shape
    buf = torch.zeros(N * ld + offset + 16, dtype=src.dtype, device=src.device)
    v = buf[offset:offset + N * ld].view(N, ld)[:, :H]
    v.copy_(src)
    return v


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H,ld,off", [(1024, 1032, 0), (1024, 1027, 0), (1024, 1024, 1), (5120, 5123, 3),
                                      (96, 100, 2), (16384, 16392, 0), (32768, 32776, 0)])
def test_strides_and_alignment(H, ld, off, dt):
    N, eps = 29, 1e-5
    t = _inputs(N, H, dt, seed=41)
    x = _strided(t["x"], ld, off)
    dy = _strided(t["dy"], ld + 8, off)
    yb = _strided(torch.zeros_like(t["x"]), ld, off)
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps, out=yb)
    dxb = _strided(torch.zeros_like(t["x"]), ld + 1, off)
    dx, dg, db = nl.ln_backward(dy, x, mean, rstd, t["gamma"], dx=dxb)
    torch.cuda.synchronize()
    xn, dyn, gn, bn = np64(t["x"]), np64(t["dy"]), np64(t["gamma"]), np64(t["beta"])
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dyn, xn, gn, eps)
    check_out(np64(y), yr, ln_y_scale(xn, mr, rr, gn, bn), dt, "strided y")
    check_out(np64(dx), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, "strided dx")
    check_param(np64(dg), dgr, dt, "strided dgamma")
    check_param(np64(db), dbr, dt, "strided dbeta")
    # the padding columns between rows stay untouched
    pad = yb.as_strided((N, ld - H), (ld, 1), yb.storage_offset() + H) if ld > H else None
    if pad is not None:
        assert torch.count_nonzero(pad[:-1]) == 0, "y padding written"
    # fused on the same layout
    r = _strided(_inputs(N, H, dt, seed=42, with_residual=True)["residual"], ld, off)
    hb = _strided(torch.zeros_like(t["x"]), ld, off)
    yf, h, _ = nl.fused_add_rms_forward(x, r, t["gamma"], 1e-6, h_out=hb)
    torch.cuda.synchronize()
    yfr, hr, rfr = O.fused_add_rms_norm_forward(xn, np64(r), gn, 1e-6, DT_ORACLE[dt])
    assert np.array_equal(np64(h), hr)
    check_out(np64(yf), yfr, rms_y_scale(xn + np64(r), rfr, gn), dt, "strided fused y")


def test_three_dim_input():
    B, T, H = 3, 17, 768
    t = _inputs(B * T, H, BF, seed=51)
    x3 = t["x"].view(B, T, H)
    y, mean, rstd = nl.ln_forward(x3, t["gamma"], t["beta"])
    assert y.shape == (B, T, H) and mean.shape == (B * T,)
    yr, _, _ = O.layer_norm_forward(np64(t["x"]), np64(t["gamma"]), np64(t["beta"]), 1e-5)
    x = np64(t["x"])
    check_bf16(np64(y).reshape(B * T, H), yr,
               ln_y_scale(x, x.mean(1), 1 / np.sqrt(x.var(1) + 1e-5), np64(t["gamma"]), np64(t["beta"])), "3-D y")


# ---------------------------------------------------------------------------
# in-place calls
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("inplace", ["x", "residual"])
@pytest.mark.parametrize("H,dt", [(4096, BF), (1000, BF), (40000, BF), (512, F32), (4096, F16)])
def test_fused_inplace(H, dt, inplace):
    fused_case(33, H, dt, seed=61, inplace=inplace)


@pytest.mark.parametrize("H,dt", [(1024, BF), (2049, F32), (16384, BF)])
def test_ln_inplace_y_and_dx(H, dt):
    N, eps = 21, 1e-5
    t = _inputs(N, H, dt, seed=71)
    xn, dyn, gn, bn = np64(t["x"]), np64(t["dy"]), np64(t["gamma"]), np64(t["beta"])
    x = t["x"].clone()
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps, out=x)
    assert y.data_ptr() == x.data_ptr()
    dy = t["dy"].clone()
    dx, dg, db = nl.ln_backward(dy, t["x"], mean, rstd, t["gamma"], dx=dy)
    torch.cuda.synchronize()
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    dxr, _, _ = O.layer_norm_backward(dyn, xn, gn, eps)
    check_out(np64(x), yr, ln_y_scale(xn, mr, rr, gn, bn), dt, "in-place y")
    check_out(np64(dy), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, "in-place dx")


# ---------------------------------------------------------------------------
# guard bands, determinism, empty inputs, error paths on the device
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, BF), (5120, BF), (16384, BF), (40000, F32), (7, F32),
                                  (5120, F16), (1000, F16)])
def test_guard_bands(H, dt):
    N, eps = 19, 1e-5
    t = _inputs(N, H, dt, seed=81)
    y = Guarded((N, H), dt, DEV)
    mean = Guarded((N,), F32, DEV)
    rstd = Guarded((N,), F32, DEV)
    lib = nl.load_library()
    code = {F32: 0, BF: 1, F16: 2}[dt]
    st = lib.ln_forward(t["x"].data_ptr(), H, t["gamma"].data_ptr(), t["beta"].data_ptr(), y.t.data_ptr(), H,
                        mean.t.data_ptr(), rstd.t.data_ptr(), N, H, eps, code, code,
                        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    dx = Guarded((N, H), dt, DEV)
    dg = Guarded((H,), dt, DEV)
    db = Guarded((H,), dt, DEV)
    wsb = nl.bwd_workspace_bytes(H)
    ws = Guarded(((wsb + 3) // 4,), F32, DEV)
    st = lib.ln_backward(t["dy"].data_ptr(), H, t["x"].data_ptr(), H, mean.t.data_ptr(), rstd.t.data_ptr(),
                         t["gamma"].data_ptr(), dx.t.data_ptr(), H, dg.t.data_ptr(), db.t.data_ptr(),
                         ws.t.data_ptr(), wsb, N, H, code, code, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    yh = Guarded((N, H), dt, DEV)
    hh = Guarded((N, H), dt, DEV)
    r = _inputs(N, H, dt, seed=82, with_residual=True)["residual"]
    st = lib.fused_add_rms_forward(t["x"].data_ptr(), H, r.data_ptr(), H, t["gamma"].data_ptr(), yh.t.data_ptr(),
                                   H, hh.t.data_ptr(), H, rstd.t.data_ptr(), N, H, 1e-6, code, code,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    for name, g in [("y", y), ("mean", mean), ("rstd", rstd), ("dx", dx), ("dgamma", dg), ("dbeta", db),
                    ("workspace", ws), ("fused y", yh), ("fused h", hh)]:
        assert g.ok(), f"{name}: write outside its buffer"


@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (2049, F32)])
def test_deterministic(H, dt):
    t = _inputs(3000, H, dt, seed=91)
    outs = []
    for _ in range(2):
        y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"])
        dx, dg, db = nl.ln_backward(t["dy"], t["x"], mean, rstd, t["gamma"])
        outs.append([a.clone() for a in (y, mean, rstd, dx, dg, db)])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8) if a.dtype == BF else a, b.view(torch.uint8) if b.dtype == BF else b)


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
def test_empty_rows(dt):
    H = 64
    x = torch.empty(0, H, dtype=dt, device=DEV)
    y, mean, rstd = nl.ln_forward(x, None, None)
    assert y.shape == (0, H)
    gamma = torch.ones(H, dtype=dt, device=DEV)
    dg0 = torch.full((H,), 5.0, dtype=dt, device=DEV)
    _, dg, db = nl.ln_backward(x, x, mean, rstd, gamma)
    _, dgr = nl.rms_backward(x, x, rstd, gamma)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dg) == 0 and torch.count_nonzero(db) == 0 and torch.count_nonzero(dgr) == 0
    del dg0


def test_device_side_errors():
    H = 256
    t = _inputs(8, H, BF, seed=3)
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"])
    small = torch.empty(16, dtype=F32, device=DEV)
    with pytest.raises(nl.NormError) as e:
        nl.ln_backward(t["dy"], t["x"], mean, rstd, t["gamma"], workspace=small)
    assert e.value.status == 3
    with pytest.raises(nl.NormError):
        nl.ln_forward(t["x"], t["gamma"], t["beta"], eps=0.0)
    # a partial overlap between h_out and x is refused
    buf = torch.zeros(9 * H, dtype=BF, device=DEV)
    xa = buf[:8 * H].view(8, H)
    hb = buf[H // 2:H // 2 + 8 * H].view(8, H)
    with pytest.raises(nl.NormError):
        nl.fused_add_rms_forward(xa, t["x"], t["gamma"], h_out=hb)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# every kernel family on the same shapes (the default policy is covered by
# every test above): 1 = register rows, 2 = strided loop, 3 = bulk-copy
# pipeline
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("path", [1, 2, 3], ids=["rows", "loop", "staged"])
@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (16384, BF), (2048, F32), (256, F32), (96, BF),
                                  (2048, F16), (16384, F16)])
def test_forced_kernel_paths(path, H, dt):
    nl._lib.set_kernel_path(path)
    try:
        ln_case(45, H, dt, seed=101 + path)
        rms_case(45, H, dt, seed=103 + path)
        fused_case(45, H, dt, seed=105 + path)
        fused_case(45, H, dt, seed=107 + path, inplace="x")
    finally:
        nl._lib.set_kernel_path(0)


def test_zz_no_device_errors():
    """No bounded wait ran out during any of the calls above."""
    torch.cuda.synchronize()
    assert nl._lib.device_errors(0, clear=True) == 0
