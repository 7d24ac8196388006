"""The allocation-free backward entry point (GPU).

ln_backward_static_workspace serves callers that cannot allocate device
memory when they call the backward; it keeps its partial sums in a scratch
array built into the library.  Through the C ABI, two calls in a row must give
what ln_backward gives with a caller-allocated workspace, within the same
tolerances as the parity tests, and a width too large for the array must be
refused.  This file is collected last so that a failure here leaves every
other test already run.
"""

import numpy as np
import pytest
import torch

import rmsnorm_ln_fwd_gb300 as nl
from normtest import check_out, check_param, ln_dx_scale, np64
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CODE = {torch.bfloat16: 1, torch.float32: 0}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def _case(N, H, dt, seed):
    c = synth.norm_inputs(N, H, "bf16" if dt == torch.bfloat16 else "f32", seed=seed)
    return {k: v.to(DEV) for k, v in c.items()}


@pytest.mark.parametrize("N,H,dt", [(2000, 1024, torch.bfloat16), (777, 5120, torch.bfloat16),
                                    (64, 256, torch.float32), (33, 1000, torch.bfloat16)])
def test_static_workspace_matches_ln_backward(N, H, dt):
    lib = nl.load_library()
    t = _case(N, H, dt, seed=N + H)
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"])
    dx_ref, dg_ref, db_ref = nl.ln_backward(t["dy"], t["x"], mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    x, dy, g = np64(t["x"]), np64(t["dy"]), np64(t["gamma"])
    for call in range(2):  # the second call reuses the array the first one left behind
        dx = torch.empty_like(t["x"])
        dg = torch.empty(H, dtype=dt, device=DEV)
        db = torch.empty(H, dtype=dt, device=DEV)
        st = lib.ln_backward_static_workspace(
            t["dy"].data_ptr(), H, t["x"].data_ptr(), H, mean.data_ptr(), rstd.data_ptr(), t["gamma"].data_ptr(),
            dx.data_ptr(), H, dg.data_ptr(), db.data_ptr(), N, H, CODE[dt], CODE[dt],
            torch.cuda.current_stream().cuda_stream)
        assert st == 0, nl._lib.status_str(st)
        torch.cuda.synchronize()
        check_out(np64(dx), np64(dx_ref), ln_dx_scale(dy, x, g, 1e-5), dt, f"call {call} dx")
        check_param(np64(dg), np64(dg_ref), dt, f"call {call} dgamma")
        check_param(np64(db), np64(db_ref), dt, f"call {call} dbeta")


def test_static_workspace_refuses_too_wide_rows():
    lib = nl.load_library()
    H = 1 << 15
    need = nl.bwd_workspace_bytes(H)
    assert need > (64 << 20)
    t = _case(2, H, torch.bfloat16, seed=1)
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"])
    dx = torch.empty_like(t["x"])
    dg = torch.empty(H, dtype=torch.bfloat16, device=DEV)
    st = lib.ln_backward_static_workspace(
        t["dy"].data_ptr(), H, t["x"].data_ptr(), H, mean.data_ptr(), rstd.data_ptr(), t["gamma"].data_ptr(),
        dx.data_ptr(), H, dg.data_ptr(), None, 2, H, 1, 1, torch.cuda.current_stream().cuda_stream)
    assert st == 3  # NORM_ERR_WORKSPACE
    torch.cuda.synchronize()
