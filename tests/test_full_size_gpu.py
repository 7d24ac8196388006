"""The measured configurations at their full sizes, in the launch configuration
the benchmark times (the auto kernel choice), against the fp64 oracle.

Every row is checked: the oracle runs over the whole input in blocks of rows
on the host, each block's row-local outputs (y, mean, rstd, dx) are compared
element by element with the kernel's, and the blocks' parameter-gradient sums
add up to the full-size dgamma/dbeta.  The fused add's stored h is checked
bit for bit everywhere.
"""

import numpy as np
import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import (DT_NAME, DT_ORACLE, check_mean, check_out, check_param, check_rstd, ln_dx_scale, ln_y_scale,
                      np64, rms_dx_scale, rms_y_scale)
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"
BF, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _blocks(N, rows=2048):
    """[i, j) row blocks covering all N rows."""
    for i in range(0, N, rows):
        yield i, min(N, i + rows)


CONFIGS = [(8192, 1024, BF), (8192, 5120, BF), (32768, 1024, BF), (16384, 2048, BF), (2048, 16384, BF),
           (512, 16384, BF), (8192, 1024, F32)]


@pytest.mark.parametrize("N,H,dt", CONFIGS, ids=[f"{n}x{h}{DT_NAME[d]}" for n, h, d in CONFIGS])
def test_ln_full_size(N, H, dt):
    eps = 1e-5
    c = synth.norm_inputs(N, H, DT_NAME[dt], seed=1)
    t = {k: v.to(DEV) for k, v in c.items()}
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"], eps)
    dx, dg, db = nl.ln_backward(t["dy"], t["x"], mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    x, dy = c["x"].double().numpy(), c["dy"].double().numpy()
    g, b = c["gamma"].double().numpy(), c["beta"].double().numpy()
    yk, mk, rk, dxk = np64(y), np64(mean), np64(rstd), np64(dx)
    dgr, dbr = np.zeros(H), np.zeros(H)
    for i, j in _blocks(N):
        xs, dys = x[i:j], dy[i:j]
        yr, mr, rr = O.layer_norm_forward(xs, g, b, eps)
        dxr, dgb, dbb = O.layer_norm_backward(dys, xs, g, eps)
        dgr += dgb
        dbr += dbb
        what = f"ln {N}x{H} rows {i}..{j - 1}"
        check_out(yk[i:j], yr, ln_y_scale(xs, mr, rr, g, b), dt, what + " y")
        check_mean(mk[i:j], mr, xs, what + " mean")
        check_rstd(rk[i:j], rr, what + " rstd")
        check_out(dxk[i:j], dxr, ln_dx_scale(dys, xs, g, eps), dt, what + " dx")
    check_param(np64(dg), dgr, dt, f"ln {N}x{H} dgamma")
    check_param(np64(db), dbr, dt, f"ln {N}x{H} dbeta")


@pytest.mark.parametrize("N,H,dt", CONFIGS, ids=[f"{n}x{h}{DT_NAME[d]}" for n, h, d in CONFIGS])
def test_rms_full_size(N, H, dt):
    eps = 1e-5
    c = synth.norm_inputs(N, H, DT_NAME[dt], seed=2, with_beta=False)
    t = {k: v.to(DEV) for k, v in c.items()}
    y, rstd = nl.rms_forward(t["x"], t["gamma"], eps)
    dx, dg = nl.rms_backward(t["dy"], t["x"], rstd, t["gamma"])
    torch.cuda.synchronize()
    x, dy, g = c["x"].double().numpy(), c["dy"].double().numpy(), c["gamma"].double().numpy()
    yk, rk, dxk = np64(y), np64(rstd), np64(dx)
    dgr = np.zeros(H)
    for i, j in _blocks(N):
        xs, dys = x[i:j], dy[i:j]
        yr, rr = O.rms_norm_forward(xs, g, eps)
        dxr, dgb = O.rms_norm_backward(dys, xs, g, eps)
        dgr += dgb
        what = f"rms {N}x{H} rows {i}..{j - 1}"
        check_out(yk[i:j], yr, rms_y_scale(xs, rr, g), dt, what + " y")
        check_rstd(rk[i:j], rr, what + " rstd")
        check_out(dxk[i:j], dxr, rms_dx_scale(dys, xs, g, eps), dt, what + " dx")
    check_param(np64(dg), dgr, dt, f"rms {N}x{H} dgamma")


def test_fused_full_size_16384x4096():
    N, H, eps = 16384, 4096, 1e-6
    c = synth.norm_inputs(N, H, "bf16", seed=3, with_beta=False, with_dy=False, with_residual=True)
    t = {k: v.to(DEV) for k, v in c.items()}
    y, h, rstd = nl.fused_add_rms_forward(t["x"], t["residual"], t["gamma"], eps)
    torch.cuda.synchronize()
    x, res, g = c["x"].double().numpy(), c["residual"].double().numpy(), c["gamma"].double().numpy()
    hn, yk, rk = np64(h), np64(y), np64(rstd)
    for i, j in _blocks(N):
        yr, hr, rr = O.fused_add_rms_norm_forward(x[i:j], res[i:j], g, eps, DT_ORACLE[BF])
        assert np.array_equal(hn[i:j], hr), f"h rows {i}..{j - 1}: not bit-exact"
        check_out(yk[i:j], yr, rms_y_scale(x[i:j] + res[i:j], rr, g), BF, f"fused y rows {i}..{j - 1}")
        check_rstd(rk[i:j], rr, f"fused rstd rows {i}..{j - 1}")


def test_fused_backward_full_size_16384x4096():
    """The fused add's backward from the stored h (with the stream gradient)."""
    N, H, eps = 16384, 4096, 1e-6
    c = synth.norm_inputs(N, H, "bf16", seed=4, with_beta=False, with_residual=True, with_dh_stream=True)
    t = {k: v.to(DEV) for k, v in c.items()}
    _, h, _ = nl.fused_add_rms_forward(t["x"], t["residual"], t["gamma"], eps)
    _, rstd_h = nl.rms_forward(h, t["gamma"], eps)   # rstd of the stored h
    dx, dres, dg = nl.fused_add_rms_backward(t["dy"], h, rstd_h, t["gamma"], t["dh_stream"])
    torch.cuda.synchronize()
    x, res = c["x"].double().numpy(), c["residual"].double().numpy()
    dy, dh, g = c["dy"].double().numpy(), c["dh_stream"].double().numpy(), c["gamma"].double().numpy()
    dxk = np64(dx)
    dgr = np.zeros(H)
    for i, j in _blocks(N):
        hs = O.round_to_dtype(O.round_to_float32(x[i:j] + res[i:j]), "bfloat16")
        dhr, dgb = O.fused_add_rms_norm_backward_from_h(dy[i:j], hs, g, eps, dh[i:j])
        dgr += dgb
        check_out(dxk[i:j], dhr, rms_dx_scale(dy[i:j], hs, g, eps) + np.abs(dh[i:j]), BF,
                  f"fused bwd dx rows {i}..{j - 1}")
    assert torch.equal(dx, dres)
    check_param(np64(dg), dgr, BF, "fused bwd dgamma")


def test_ln_backward_from_output_full_size_8192x5120():
    """The backward from the saved output at full size.  Its inputs y and
    rstd are drawn from the generator (any y and positive rstd are valid
    inputs), and both sides take the same values."""
    N, H = 8192, 5120
    c = synth.norm_inputs(N, H, "bf16", seed=5)
    t = {k: v.to(DEV) for k, v in c.items()}
    rstd = (0.5 + synth.normal((N,), 5, "residual").abs()).to(DEV)
    dx, dg, db = nl.ln_backward_from_output(t["dy"], t["x"], rstd, t["gamma"], t["beta"])
    torch.cuda.synchronize()
    y, dy = c["x"].double().numpy(), c["dy"].double().numpy()
    g, b, r = c["gamma"].double().numpy(), c["beta"].double().numpy(), np64(rstd)
    dxk = np64(dx)
    dgr, dbr = np.zeros(H), np.zeros(H)
    for i, j in _blocks(N):
        dxr, dgb, dbb = O.layer_norm_backward_from_output(dy[i:j], y[i:j], r[i:j], g, b)
        dgr += dgb
        dbr += dbb
        xh = (y[i:j] - b) / g
        gg = dy[i:j] * g
        scale = r[i:j, None] * (np.abs(gg) + np.abs(gg).mean(1, keepdims=True) +
                                np.abs(xh) * np.abs(gg * xh).mean(1, keepdims=True))
        check_out(dxk[i:j], dxr, scale, BF, f"from-output dx rows {i}..{j - 1}")
    check_param(np64(dg), dgr, BF, "from-output dgamma")
    check_param(np64(db), dbr, BF, "from-output dbeta")


def test_beyond_2pow31_elements():
    """N*H just past 2^31 elements (bf16, H = 1024): row offsets need 64-bit
    arithmetic.  The rows repeat a seeded 4096-row block, so the oracle works
    on that block: sampled rows (the last ones among them) row by row, and the
    parameter gradients as block sums weighted by how often each row occurs."""
    H, B, eps = 1024, 4096, 1e-5
    N = (1 << 31) // H + 3
    c = synth.norm_inputs(B, H, "bf16", seed=6)
    reps = (N + B - 1) // B
    x = c["x"].to(DEV).repeat(reps, 1)[:N]
    dy = c["dy"].to(DEV).repeat(reps, 1)[:N]
    gamma, beta = c["gamma"].to(DEV), c["beta"].to(DEV)
    y, mean, rstd = nl.ln_forward(x, gamma, beta, eps)
    dx, dg, db = nl.ln_backward(dy, x, mean, rstd, gamma)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, N - 1, N - 2, N - 3], np.random.default_rng(12).choice(N, 28)]))
    idx = torch.as_tensor(rows, device=DEV)
    xb, dyb = c["x"].double().numpy(), c["dy"].double().numpy()
    g, b = c["gamma"].double().numpy(), c["beta"].double().numpy()
    xs, dys = xb[rows % B], dyb[rows % B]
    yr, mr, rr = O.layer_norm_forward(xs, g, b, eps)
    dxr, _, _ = O.layer_norm_backward(dys, xs, g, eps)
    check_out(np64(y.index_select(0, idx)), yr, ln_y_scale(xs, mr, rr, g, b), BF, "2^31 y rows")
    check_rstd(np64(rstd.index_select(0, idx)), rr, "2^31 rstd rows")
    check_out(np64(dx.index_select(0, idx)), dxr, ln_dx_scale(dys, xs, g, eps), BF, "2^31 dx rows")
    # Every other row: a row's outputs depend on that row alone, and the rows
    # repeat the block, so each later block must equal the first bit for bit
    # (the first block's last rows are among the sampled rows above).
    for out in (y, mean, rstd, dx):
        first = out[:B]
        for i in range(B, N, B):
            j = min(N, i + B)
            assert torch.equal(out[i:j], first[:j - i]), f"2^31 rows {i}..{j - 1} differ from the first block"
    count = np.full(B, N // B, dtype=np.float64)
    count[:N % B] += 1
    _, dgb, dbb = O.layer_norm_backward(dyb * count[:, None], xb, g, eps)
    check_param(np64(dg), dgb, BF, "2^31 dgamma")
    check_param(np64(db), dbb, BF, "2^31 dbeta")
