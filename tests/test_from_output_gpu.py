"""LayerNorm / RMSNorm backward from the forward's saved output, CUDA path vs
the fp64 oracle ("Rewrite Triton normalization backward kernel_1 (#499)",
Benchmark harness: the backward reads the saved output).

The backward is a function of (dy, y, rstd, gamma, beta), so most cases draw
those directly from the seeded generator and hand the same values to both
sides.  The training-chain case runs the forward first and compares against
the oracle's backward from x, with the bound widened by what the rounding of
the stored y can move x_hat = (y - beta)/gamma.
"""

import numpy as np
import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import DT_NAME, Guarded, bf16_ulp, check_out, check_param, f16_ulp, ln_y_scale, np64
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF, F32, F16 = torch.bfloat16, torch.float32, torch.float16
DTS, DT_IDS = [BF, F32, F16], ["bf16", "f32", "f16"]
CODE = {F32: 0, BF: 1, F16: 2}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _inputs(N, H, dt, seed, wdt=None):
    """dy, gamma, beta and a y of the forward's typical size from the
    generator; rstd = 0.5 + |N(0,1)| (any positive value is a valid input)."""
    d = synth.norm_inputs(N, H, DT_NAME[dt], None if wdt is None else DT_NAME[wdt], seed)
    t = {k: v.to(DEV) for k, v in d.items()}
    t["y"] = t.pop("x")
    t["rstd"] = (0.5 + synth.normal((N,), seed, "residual").abs()).to(DEV)
    return t


def _dx_scale(dy, xh, gamma, rstd, ln):
    """Magnitude of what dx_i = rstd*(g_i - c1 - x_hat_i*c2) is formed from."""
    H = dy.shape[1]
    g = dy * (np.ones(H) if gamma is None else gamma)
    c1 = np.abs(g).mean(axis=1, keepdims=True) if ln else 0.0
    c2 = np.abs(g * xh).mean(axis=1, keepdims=True)
    return rstd[:, None] * (np.abs(g) + c1 + np.abs(xh) * c2)


def _x_hat(y, gamma, beta):
    H = y.shape[1]
    g = np.ones(H) if gamma is None else gamma
    b = np.zeros(H) if beta is None else beta
    return (y - b) / g


def ln_y_case(N, H, dt, seed=0, gamma=True, beta=True, wdt=None, dx_into_dy=False):
    t = _inputs(N, H, dt, seed, wdt)
    g = t["gamma"] if gamma else None
    b = t["beta"] if beta else None
    dy0 = t["dy"].clone()
    dx, dg, db = nl.ln_backward_from_output(t["dy"], t["y"], t["rstd"], g, b, dx=t["dy"] if dx_into_dy else None)
    torch.cuda.synchronize()
    dyn, yn, rn = np64(dy0), np64(t["y"]), np64(t["rstd"])
    gn = None if g is None else np64(g)
    bn = None if b is None else np64(b)
    dxr, dgr, dbr = O.layer_norm_backward_from_output(dyn, yn, rn, gn, bn)
    xh = _x_hat(yn, gn, bn)
    what = f"ln from y {N}x{H} {DT_NAME[dt]}"
    check_out(np64(dx), dxr, _dx_scale(dyn, xh, gn, rn, True), dt, what + " dx")
    check_param(np64(dg), dgr, dg.dtype, what + " dgamma")
    check_param(np64(db), dbr, db.dtype, what + " dbeta")
    if not dx_into_dy:
        assert torch.equal(t["dy"], dy0), "dy modified"


def rms_y_case(N, H, dt, seed=0, gamma=True, wdt=None, dx_into_dy=False):
    t = _inputs(N, H, dt, seed, wdt)
    g = t["gamma"] if gamma else None
    dy0 = t["dy"].clone()
    dx, dg = nl.rms_backward_from_output(t["dy"], t["y"], t["rstd"], g, dx=t["dy"] if dx_into_dy else None)
    torch.cuda.synchronize()
    dyn, yn, rn = np64(dy0), np64(t["y"]), np64(t["rstd"])
    gn = None if g is None else np64(g)
    dxr, dgr = O.rms_norm_backward_from_output(dyn, yn, rn, gn)
    xh = _x_hat(yn, gn, None)
    what = f"rms from y {N}x{H} {DT_NAME[dt]}"
    check_out(np64(dx), dxr, _dx_scale(dyn, xh, gn, rn, False), dt, what + " dx")
    check_param(np64(dg), dgr, dg.dtype, what + " dgamma")


H_SWEEP = [1, 7, 8, 32, 33, 64, 256, 1000, 1024, 2049, 4096, 5120, 8192, 16384, 40000]


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H", H_SWEEP)
def test_ln_from_output_sweep(H, dt):
    ln_y_case(37, H, dt, seed=H)


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
@pytest.mark.parametrize("H", H_SWEEP)
def test_rms_from_output_sweep(H, dt):
    rms_y_case(37, H, dt, seed=H + 1)


@pytest.mark.parametrize("N", [1, 2, 153, 1000, 5000])
@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (2048, F32), (4096, F16)])
def test_from_output_row_counts(N, H, dt):
    ln_y_case(N, H, dt, seed=N)
    rms_y_case(N, H, dt, seed=N + 1)


@pytest.mark.parametrize("H,dt", [(1024, BF), (33, F32), (5120, F16)])
def test_from_output_without_affine(H, dt):
    ln_y_case(29, H, dt, seed=3, gamma=False, beta=False)
    ln_y_case(29, H, dt, seed=4, gamma=True, beta=False)
    ln_y_case(29, H, dt, seed=5, gamma=False, beta=True)
    rms_y_case(29, H, dt, seed=6, gamma=False)


@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, F16), (5120, BF), (16384, BF), (32768, F16)])
def test_from_output_fp32_params(H, dt):
    ln_y_case(29, H, dt, seed=7, wdt=F32)
    rms_y_case(29, H, dt, seed=8, wdt=F32)


@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, BF), (16384, BF), (512, F32)])
def test_from_output_dx_in_place(H, dt):
    ln_y_case(29, H, dt, seed=9, dx_into_dy=True)
    rms_y_case(29, H, dt, seed=10, dx_into_dy=True)


@pytest.mark.parametrize("path", [1, 2, 3], ids=["rows", "loop", "staged"])
@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (16384, BF), (2048, F32), (96, BF), (4096, F16)])
def test_from_output_forced_paths(path, H, dt):
    nl._lib.set_kernel_path(path)
    try:
        ln_y_case(41, H, dt, seed=11)
        rms_y_case(41, H, dt, seed=12)
    finally:
        nl._lib.set_kernel_path(0)


def _strided(src, ld, offset=0):
    N, H = src.shape
    buf = torch.zeros(N * ld + offset + H, dtype=src.dtype, device=src.device)
    v = buf[offset:offset + N * ld].view(N, ld)[:, :H]
    v.copy_(src)
    return v


@pytest.mark.parametrize("H,ld,off,dt", [(1024, 1032, 0, BF), (1024, 1027, 0, BF), (1024, 1024, 1, BF),
                                         (5120, 5123, 3, F16), (2048, 2049, 0, F32), (16384, 16392, 0, BF)])
def test_from_output_strides_and_alignment(H, ld, off, dt):
    N = 29
    t = _inputs(N, H, dt, 13)
    y, dy = _strided(t["y"], ld, off), _strided(t["dy"], ld + 8, off)
    dxb = _strided(torch.zeros_like(t["y"]), ld + 1, off)
    dx, dg, db = nl.ln_backward_from_output(dy, y, t["rstd"], t["gamma"], t["beta"], dx=dxb)
    torch.cuda.synchronize()
    dyn, yn, rn, gn, bn = np64(t["dy"]), np64(t["y"]), np64(t["rstd"]), np64(t["gamma"]), np64(t["beta"])
    dxr, dgr, dbr = O.layer_norm_backward_from_output(dyn, yn, rn, gn, bn)
    check_out(np64(dx), dxr, _dx_scale(dyn, _x_hat(yn, gn, bn), gn, rn, True), dt, "strided dx")
    check_param(np64(dg), dgr, dt, "strided dgamma")
    check_param(np64(db), dbr, dt, "strided dbeta")


@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, BF), (5120, BF), (40000, F32), (7, F32), (4096, F16)])
def test_from_output_guard_bands(H, dt):
    N = 19
    t = _inputs(N, H, dt, 15)
    gx, gg, gb = Guarded((N, H), dt, DEV), Guarded((H,), dt, DEV), Guarded((H,), dt, DEV)
    lib = nl._lib.load()
    ws_bytes = nl.bwd_workspace_bytes(H)
    ws = torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=DEV)
    st = lib.ln_backward_from_output(t["dy"].data_ptr(), H, t["y"].data_ptr(), H, t["rstd"].data_ptr(),
                                     t["gamma"].data_ptr(), t["beta"].data_ptr(), gx.t.data_ptr(), H,
                                     gg.t.data_ptr(), gb.t.data_ptr(), ws.data_ptr(), ws_bytes, N, H, CODE[dt],
                                     CODE[dt], torch.cuda.current_stream().cuda_stream)
    nl._lib.check("ln_backward_from_output", st)
    torch.cuda.synchronize()
    assert gx.ok() and gg.ok() and gb.ok(), "write outside an output"
    dyn, yn, rn, gn, bn = np64(t["dy"]), np64(t["y"]), np64(t["rstd"]), np64(t["gamma"]), np64(t["beta"])
    dxr, dgr, dbr = O.layer_norm_backward_from_output(dyn, yn, rn, gn, bn)
    check_out(np64(gx.t), dxr, _dx_scale(dyn, _x_hat(yn, gn, bn), gn, rn, True), dt, "guarded dx")
    check_param(np64(gg.t), dgr, dt, "guarded dgamma")
    check_param(np64(gb.t), dbr, dt, "guarded dbeta")


@pytest.mark.parametrize("H,dt", [(1024, BF), (4096, BF), (5120, BF), (1000, F32), (2048, F16)])
def test_from_output_training_chain(H, dt):
    """Forward, then the backward from its stored y and saved rstd, against the
    oracle's backward from x.  y_stored is within one ulp plus the fp32 slack of
    the exact output; that error divided by |gamma| bounds the error delta of
    the recovered x_hat, and dx = rstd*(g - c1 - x_hat*c2) then moves by at most
    rstd*(delta*|c2| + |x_hat|*mean(|g|*delta) + delta*mean(|g|*delta))."""
    N, eps = 64, 1e-5
    d = synth.norm_inputs(N, H, DT_NAME[dt], None, 17)
    t = {k: v.to(DEV) for k, v in d.items()}
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"], eps)
    dx, dg, db = nl.ln_backward_from_output(t["dy"], y, rstd, t["gamma"], t["beta"])
    torch.cuda.synchronize()
    x, dyn, gn, bn = np64(t["x"]), np64(t["dy"]), np64(t["gamma"]), np64(t["beta"])
    yr, mr, rr = O.layer_norm_forward(x, gn, bn, eps)
    dxr, dgr, dbr = O.layer_norm_backward(dyn, x, gn, eps)
    xh = (x - mr[:, None]) * rr[:, None]
    ulp = {BF: bf16_ulp, F16: f16_ulp, F32: lambda r: np.abs(r) * 2.0 ** -23}[dt]
    e_y = ulp(yr) + 2.0 ** -20 * ln_y_scale(x, mr, rr, gn, bn)
    delta = e_y / np.abs(gn) + 2.0 ** -22 * np.abs(xh)
    g = dyn * gn
    c2 = np.abs(g * xh).mean(axis=1, keepdims=True)
    mgd = (np.abs(g) * delta).mean(axis=1, keepdims=True)
    move = rr[:, None] * (delta * c2 + np.abs(xh) * mgd + delta * mgd)
    base = _dx_scale(dyn, xh, gn, rr, True)
    if dt == F32:
        err = np.max(np.abs(np64(dx) - dxr))
        assert err <= 1e-5 * np.max(np.abs(dxr)) + np.max(move), f"chain dx: {err:.3e}"
    else:
        check_out(np64(dx), dxr, base + move * 2.0 ** 20, dt, "chain dx")
    dg_move = (np.abs(dyn) * delta).sum(axis=0)
    e = np.linalg.norm(np64(dg) - dgr) / np.linalg.norm(dgr)
    bound = (1e-5 if dt == F32 else 5e-3) + np.linalg.norm(dg_move) / np.linalg.norm(dgr)
    assert e <= bound, f"chain dgamma: relative RMS {e:.3e} > {bound:.3e}"
    check_param(np64(db), dbr, db.dtype, "chain dbeta")


@pytest.mark.parametrize("dt", DTS, ids=DT_IDS)
def test_from_output_empty_rows(dt):
    H = 256
    y = torch.empty(0, H, dtype=dt, device=DEV)
    rstd = torch.empty(0, dtype=torch.float32, device=DEV)
    gamma = torch.ones(H, dtype=dt, device=DEV)
    dx, dg, db = nl.ln_backward_from_output(y.clone(), y, rstd, gamma, gamma)
    dxr, dgr = nl.rms_backward_from_output(y.clone(), y, rstd, gamma)
    torch.cuda.synchronize()
    assert dx.shape == (0, H) and dxr.shape == (0, H)
    assert torch.count_nonzero(dg).item() == 0 and torch.count_nonzero(db).item() == 0
    assert torch.count_nonzero(dgr).item() == 0


def test_from_output_zz_no_device_errors():
    assert nl._lib.device_errors(0, clear=True) == 0
