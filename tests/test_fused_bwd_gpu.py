"""Fused residual add + RMSNorm backward, CUDA path vs the fp64 oracle.

The backward reads the stored sum h and its rstd and returns dL/dh, the
gradient of both x and the residual, plus the gradient arriving through h
itself when one is given ("Skill: Write a Triton Fused Add+RMSNorm Kernel",
Required reasoning process steps 9-10).

Most cases give the kernel rstd of the stored h (an RMSNorm forward of h),
so kernel and oracle differentiate at the same point.  In training the saved
rstd comes from the fp32 sum before h was rounded to bf16; the training-chain
case widens the bf16 bound by the measured per-row rstd difference.
"""

import numpy as np
import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import DT_NAME, DT_ORACLE, Guarded, check_out, check_param, np64, rms_dx_scale
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF, F32, F16 = torch.bfloat16, torch.float32, torch.float16
CODE = {F32: 0, BF: 1, F16: 2}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _inputs(N, H, dt, seed):
    d = synth.norm_inputs(N, H, DT_NAME[dt], None, seed, with_beta=False,
                          with_residual=True, with_dh_stream=True)
    return {k: v.to(DEV) for k, v in d.items()}


def _stored_h(t, eps):
    """h and rstd as the training forward leaves them, and the oracle's own h
    and rstd (the oracle side never takes an input from the CUDA path; the two
    h agree bit for bit, which is checked here)."""
    _, h, rstd = nl.fused_add_rms_forward(t["x"], t["residual"], t["gamma"], eps)
    torch.cuda.synchronize()
    _, hr, rr = O.fused_add_rms_norm_forward(np64(t["x"]), np64(t["residual"]), np64(t["gamma"]), eps,
                                             DT_ORACLE[h.dtype])
    assert np.array_equal(np64(h), hr), "stored h differs from the oracle's"
    return h, rstd, hr, rr


def fused_bwd_case(N, H, dt, eps=1e-6, seed=0, with_dh=True, residual_grad="separate", dx_into=None,
                   saved_rstd=False, gamma=True):
    t = _inputs(N, H, dt, seed)
    h, rstd_fwd, hn, rr = _stored_h(t, eps)
    g = t["gamma"] if gamma else None
    # rstd of the stored h itself (the training forward's rstd is of the
    # unrounded fp32 sum; identical for fp32 rows)
    rstd = rstd_fwd if saved_rstd else nl.rms_forward(h, g if g is not None else None, eps)[1]
    dy = t["dy"]
    dh = t["dh_stream"] if with_dh else None
    dy0 = dy.clone()
    dh0 = None if dh is None else dh.clone()
    dx_buf = {None: None, "dy": dy, "dh": dh}[dx_into]
    dx, dres, dg = nl.fused_add_rms_backward(dy, h, rstd, g, dh, residual_grad=residual_grad, dx=dx_buf)
    torch.cuda.synchronize()

    dyn = np64(dy0)
    gn = None if g is None else np64(g)
    dhn = None if dh0 is None else np64(dh0)
    dhr, dgr = O.fused_add_rms_norm_backward_from_h(dyn, hn, gn, eps, dhn)
    mult = 2.0 if residual_grad == "same" else 1.0
    scale = rms_dx_scale(dyn, hn, gn, eps)
    if dhn is not None:
        scale = scale + np.abs(dhn)
    if saved_rstd and dt != F32:
        # dx = rstd*g - rstd^3*h*sum(g*h)/H: a relative rstd difference d per
        # row moves dx by at most 3*d times its terms' magnitude.  d is the
        # oracle's: rstd of the exact sum against rstd of the stored h (the
        # saved fp32 rstd sits within 2^-22 of the former).
        r_h = O.rms_norm_forward(hn, None, eps)[1]
        d = np.abs(rr / r_h - 1.0) + 2.0 ** -22
        scale = scale * (1.0 + 3.0 * d[:, None] * 2.0 ** 20)
    what = f"fused bwd {N}x{H} dh={with_dh} res={residual_grad} into={dx_into}"
    check_out(np64(dx), mult * dhr, mult * scale, dt, what + " dx")
    if residual_grad == "separate":
        assert torch.equal(dres, dx), what + ": dres differs from dx"
    elif residual_grad == "same":
        assert dres is dx
    else:
        assert dres is None
    if dg is not None:
        check_param(np64(dg), dgr, dg.dtype, what + " dgamma")
    if dx_into != "dy":
        assert torch.equal(dy, dy0), "dy modified"
    if dh is not None and dx_into != "dh":
        assert torch.equal(dh, dh0), "dh_stream modified"


H_SWEEP = [1, 7, 8, 32, 33, 64, 256, 1000, 1024, 2049, 4096, 5120, 8192, 12288, 16384, 40000]


@pytest.mark.parametrize("dt", [BF, F32, F16], ids=["bf16", "f32", "f16"])
@pytest.mark.parametrize("H", H_SWEEP)
def test_fused_bwd_sweep(H, dt):
    fused_bwd_case(37 if H > 8192 else 67, H, dt)


@pytest.mark.parametrize("dt", [BF, F32], ids=["bf16", "f32"])
@pytest.mark.parametrize("H", [1024, 1000, 5120])
def test_fused_bwd_without_stream_gradient(H, dt):
    fused_bwd_case(67, H, dt, with_dh=False)


@pytest.mark.parametrize("mode", ["separate", "none", "same"])
@pytest.mark.parametrize("H,dt", [(1024, BF), (4096, BF), (1000, BF), (2048, F32), (7, F32), (16384, BF),
                                  (32768, BF)])
def test_fused_bwd_residual_grad_modes(mode, H, dt):
    fused_bwd_case(67, H, dt, residual_grad=mode)


@pytest.mark.parametrize("into", ["dy", "dh"])
@pytest.mark.parametrize("mode", ["separate", "none", "same"])
@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, BF), (16384, BF), (512, F32), (2048, F16)])
def test_fused_bwd_in_place(into, mode, H, dt):
    fused_bwd_case(67, H, dt, residual_grad=mode, dx_into=into)


@pytest.mark.parametrize("N", [1, 2, 153, 1000, 5000])
@pytest.mark.parametrize("H,dt", [(4096, BF), (1024, BF), (2048, F32)])
def test_fused_bwd_row_counts(N, H, dt):
    fused_bwd_case(N, H, dt)


@pytest.mark.parametrize("H,dt", [(1024, BF), (4096, BF), (5120, BF), (1000, F32), (2048, F32), (1024, F16),
                                  (4096, F16)])
def test_fused_bwd_training_chain(H, dt):
    """Forward then backward with the forward's own saved rstd."""
    fused_bwd_case(200, H, dt, saved_rstd=True)


@pytest.mark.parametrize("H,dt", [(1024, BF), (33, F32)])
def test_fused_bwd_no_gamma(H, dt):
    fused_bwd_case(67, H, dt, gamma=False)


@pytest.mark.parametrize("path", [1, 2, 3], ids=["rows", "loop", "staged"])
@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (16384, BF), (2048, F32), (96, BF)])
def test_fused_bwd_forced_paths(path, H, dt):
    nl._lib.set_kernel_path(path)
    try:
        fused_bwd_case(67, H, dt)
        fused_bwd_case(67, H, dt, residual_grad="same", with_dh=False)
    finally:
        nl._lib.set_kernel_path(0)


def _strided(src, ld, offset=0):
    N, H = src.shape
    buf = torch.zeros(N * ld + offset + H, dtype=src.dtype, device=src.device)
    v = buf[offset:offset + N * ld].view(N, ld)[:, :H]
    v.copy_(src)
    return v


@pytest.mark.parametrize("H,ld,off,dt", [(1024, 1032, 0, BF), (1024, 1027, 0, BF), (1024, 1024, 1, BF),
                                         (5120, 5123, 3, BF), (2048, 2049, 0, F32), (16384, 16392, 0, BF)])
def test_fused_bwd_strides_and_alignment(H, ld, off, dt):
    N, eps = 67, 1e-6
    t = _inputs(N, H, dt, 3)
    h, _, hn, _ = _stored_h(t, eps)
    rstd = nl.rms_forward(h, t["gamma"], eps)[1]
    dy, hs, dh = _strided(t["dy"], ld, off), _strided(h, ld, off), _strided(t["dh_stream"], ld, off)
    dxs = _strided(torch.zeros_like(h), ld, off)
    drs = _strided(torch.zeros_like(h), ld + 8, off)
    lib = nl._lib.load()
    ws_bytes = nl.bwd_workspace_bytes(H)
    ws = torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=DEV)
    dg = torch.empty(H, dtype=dt, device=DEV)
    code = CODE[dt]
    st = lib.fused_add_rms_backward(dy.data_ptr(), ld, hs.data_ptr(), ld, rstd.data_ptr(), t["gamma"].data_ptr(),
                                    dh.data_ptr(), ld, dxs.data_ptr(), ld, drs.data_ptr(), ld + 8, dg.data_ptr(),
                                    ws.data_ptr(), ws_bytes, N, H, code, code,
                                    torch.cuda.current_stream().cuda_stream)
    nl._lib.check("fused_add_rms_backward", st)
    torch.cuda.synchronize()
    dyn, dhn, gn = np64(t["dy"]), np64(t["dh_stream"]), np64(t["gamma"])
    dhr, dgr = O.fused_add_rms_norm_backward_from_h(dyn, hn, gn, eps, dhn)
    scale = rms_dx_scale(dyn, hn, gn, eps) + np.abs(dhn)
    check_out(np64(dxs), dhr, scale, dt, f"strided dx {H}/{ld}+{off}")
    assert torch.equal(dxs, drs), "dres differs from dx"
    check_param(np64(dg), dgr, dt, f"strided dgamma {H}/{ld}+{off}")


@pytest.mark.parametrize("H,dt", [(1024, BF), (1000, BF), (16384, BF), (40000, F32), (7, F32), (4096, F16)])
def test_fused_bwd_guard_bands(H, dt):
    N, eps = 67, 1e-6
    t = _inputs(N, H, dt, 5)
    h, _, hn, _ = _stored_h(t, eps)
    rstd = nl.rms_forward(h, t["gamma"], eps)[1]
    gx, gr, gg = Guarded((N, H), dt, DEV), Guarded((N, H), dt, DEV), Guarded((H,), dt, DEV)
    lib = nl._lib.load()
    ws_bytes = nl.bwd_workspace_bytes(H)
    ws = torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=DEV)
    code = CODE[dt]
    st = lib.fused_add_rms_backward(t["dy"].data_ptr(), H, h.data_ptr(), H, rstd.data_ptr(), t["gamma"].data_ptr(),
                                    t["dh_stream"].data_ptr(), H, gx.t.data_ptr(), H, gr.t.data_ptr(), H,
                                    gg.t.data_ptr(), ws.data_ptr(), ws_bytes, N, H, code, code,
                                    torch.cuda.current_stream().cuda_stream)
    nl._lib.check("fused_add_rms_backward", st)
    torch.cuda.synchronize()
    assert gx.ok() and gr.ok() and gg.ok(), "write outside an output"
    dyn, dhn, gn = np64(t["dy"]), np64(t["dh_stream"]), np64(t["gamma"])
    dhr, dgr = O.fused_add_rms_norm_backward_from_h(dyn, hn, gn, eps, dhn)
    check_out(np64(gx.t), dhr, rms_dx_scale(dyn, hn, gn, eps) + np.abs(dhn), dt, f"guarded dx {H}")
    assert torch.equal(gx.t, gr.t)
    check_param(np64(gg.t), dgr, dt, f"guarded dgamma {H}")


@pytest.mark.parametrize("H,dt", [(1024, BF), (5120, BF), (2049, F32)])
def test_fused_bwd_deterministic(H, dt):
    t = _inputs(300, H, dt, 7)
    h, rstd, _, _ = _stored_h(t, 1e-6)
    a = nl.fused_add_rms_backward(t["dy"], h, rstd, t["gamma"], t["dh_stream"])
    b = nl.fused_add_rms_backward(t["dy"], h, rstd, t["gamma"], t["dh_stream"])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("dt", [BF, F32], ids=["bf16", "f32"])
def test_fused_bwd_empty_rows(dt):
    H = 256
    h = torch.empty(0, H, dtype=dt, device=DEV)
    dy = torch.empty(0, H, dtype=dt, device=DEV)
    rstd = torch.empty(0, dtype=torch.float32, device=DEV)
    gamma = torch.ones(H, dtype=dt, device=DEV)
    dx, dres, dg = nl.fused_add_rms_backward(dy, h, rstd, gamma, None)
    torch.cuda.synchronize()
    assert dx.shape == (0, H) and dres.shape == (0, H)
    assert torch.count_nonzero(dg).item() == 0


def test_fused_bwd_zz_no_device_errors():
    assert nl._lib.device_errors(0, clear=True) == 0
