"""The span-row backward kernels at their boundaries, against the fp64 oracle.

Half-precision LayerNorm rows of at most 256 threads (16 contiguous columns a
thread, H a multiple of 16, rows 32-byte aligned) take the span kernel with a
register prefetch; LayerNorm and RMSNorm rows of 257..640 threads take span
rows whose next rows are bulk-copied into shared memory.  The cases straddle
those limits (4096 = 256 threads, 4112 = 257, 10240 = 640, 10256 = 641), run
ragged and tiny row counts (fewer rows than CTAs, a last partial wave), padded
strides that keep 32-byte alignment (the span paths) and strides that keep
only 16-byte alignment (the interleaved register rows), the saved statistics
of the GPU forward, and both dgamma/dbeta requested and dx alone; and the
backward from the forward's saved output on the shared-memory span rows.
"""

import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import DT_NAME, check_out, check_param, ln_dx_scale, ln_y_scale, np64, rms_dx_scale
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF, F16 = torch.bfloat16, torch.float16


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


def _run(kind, N, H, dt, ld=None, param_grads=True, seed=3):
    eps = 1e-5
    t = {k: v.to(DEV) for k, v in synth.norm_inputs(N, H, DT_NAME[dt], seed=seed).items()}
    x, dy = t["x"], t["dy"]
    if ld is not None:
        x, dy = _strided(x, ld), _strided(dy, ld)
    g = t["gamma"]
    xn, dyn, gn = np64(t["x"]), np64(t["dy"]), np64(g)
    dxb = _strided(torch.zeros_like(t["x"]), ld) if ld is not None else None
    if kind == "ln":
        _, mean, rstd = nl.ln_forward(x, g, t["beta"], eps)
        dx, dg, db = nl.ln_backward(dy, x, mean, rstd, g, dx=dxb, need_param_grads=param_grads)
        torch.cuda.synchronize()
        dxr, dgr, dbr = O.layer_norm_backward(dyn, xn, gn, eps)
        check_out(np64(dx), dxr, ln_dx_scale(dyn, xn, gn, eps), dt, f"ln dx {N}x{H} ld={ld}")
        if param_grads:
            check_param(np64(dg), dgr, dt, f"ln dgamma {N}x{H}")
            check_param(np64(db), dbr, dt, f"ln dbeta {N}x{H}")
    else:
        _, rstd = nl.rms_forward(x, g, eps)
        dx, dg = nl.rms_backward(dy, x, rstd, g, dx=dxb, need_param_grads=param_grads)
        torch.cuda.synchronize()
        dxr, dgr = O.rms_norm_backward(dyn, xn, gn, eps)
        check_out(np64(dx), dxr, rms_dx_scale(dyn, xn, gn, eps), dt, f"rms dx {N}x{H} ld={ld}")
        if param_grads:
            check_param(np64(dg), dgr, dt, f"rms dgamma {N}x{H}")
    if ld is not None and ld > H:  # the padding between rows stays untouched
        pad = dxb.as_strided((N - 1, ld - H), (ld, 1), dxb.storage_offset() + H)
        assert torch.count_nonzero(pad) == 0, "dx padding written"


@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [512, 2048, 4096, 4112, 5120, 8192, 10240, 10256])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_span_widths(kind, H, dt):
    _run(kind, 700, H, dt)


@pytest.mark.parametrize("N", [1, 7, 151, 305, 2049])
@pytest.mark.parametrize("H", [1024, 5120])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_span_row_counts(kind, N, H):
    _run(kind, N, H, BF, seed=N)


@pytest.mark.parametrize("H,ld", [(1024, 1040), (1024, 1032), (5120, 5136), (5120, 5128), (4112, 4128)])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_span_strides(kind, H, ld):
    # ld - H = 16 elements keeps every row 32-byte aligned (span paths); 8
    # keeps 16-byte alignment only (interleaved register rows)
    _run(kind, 333, H, BF, ld=ld)


@pytest.mark.parametrize("H", [1024, 5120])
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_span_dx_only(kind, H):
    _run(kind, 500, H, BF, param_grads=False)


# The backward from the forward's saved output on the span rows from shared
# memory (rows of 257..640 threads): x_hat = (y - beta)/gamma from per-thread
# 1/gamma and beta slots, next to gamma.
from test_from_output_gpu import ln_y_case, rms_y_case  # noqa: E402


@pytest.mark.parametrize("dt", [BF, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [4096, 4112, 5120, 8192, 10240, 10256])
def test_span_from_output_widths(H, dt):
    ln_y_case(300, H, dt, seed=H)
    rms_y_case(300, H, dt, seed=H + 1)


@pytest.mark.parametrize("N", [1, 7, 305])
def test_span_from_output_row_counts_and_params(N):
    ln_y_case(N, 5120, BF, seed=N)
    rms_y_case(N, 5120, BF, seed=N + 1)
    ln_y_case(N, 5120, BF, seed=N + 2, wdt=torch.float32)      # fp32 parameters
    ln_y_case(N, 5120, F16, seed=N + 3, gamma=False, beta=False)  # no affine
    rms_y_case(N, 5120, F16, seed=N + 4, gamma=False)


@pytest.mark.parametrize("H", [5120, 8192])
def test_span_in_place(H):
    """y over x in the forward (wide-chunk rows) and dx over dy in the
    backward (span rows from shared memory, from x and from the output): each
    row's dy sits in shared memory before that row's dx is written."""
    N, eps = 333, 1e-5
    t = {k: v.to(DEV) for k, v in synth.norm_inputs(N, H, "bf16", seed=H).items()}
    xn, dyn, gn, bn = np64(t["x"]), np64(t["dy"]), np64(t["gamma"]), np64(t["beta"])
    x = t["x"].clone()
    y, mean, rstd = nl.ln_forward(x, t["gamma"], t["beta"], eps, out=x)
    assert y.data_ptr() == x.data_ptr()
    dy = t["dy"].clone()
    nl.ln_backward(dy, t["x"], mean, rstd, t["gamma"], dx=dy)
    dy2 = t["dy"].clone()
    _, rstd2 = nl.rms_forward(t["x"], t["gamma"], eps)
    nl.rms_backward(dy2, t["x"], rstd2, t["gamma"], dx=dy2)
    torch.cuda.synchronize()
    yr, mr, rr = O.layer_norm_forward(xn, gn, bn, eps)
    check_out(np64(x), yr, ln_y_scale(xn, mr, rr, gn, bn), BF, f"in-place y {H}")
    dxr, _, _ = O.layer_norm_backward(dyn, xn, gn, eps)
    check_out(np64(dy), dxr, ln_dx_scale(dyn, xn, gn, eps), BF, f"in-place ln dx {H}")
    dxr2, _ = O.rms_norm_backward(dyn, xn, gn, eps)
    check_out(np64(dy2), dxr2, rms_dx_scale(dyn, xn, gn, eps), BF, f"in-place rms dx {H}")
    ln_y_case(N, H, BF, seed=H + 5, dx_into_dy=True)
    rms_y_case(N, H, BF, seed=H + 6, dx_into_dy=True)
