"""The allocation-free backward entry point (GPU).

ln_backward_static_workspace serves callers that cannot allocate device
memory when they call the backward; it keeps its partial sums in a scratch
array built into the library.  Through the C ABI, two calls in a row must
match the fp64 oracle and what ln_backward gives with a caller-allocated
workspace, within the same tolerances as the parity tests (the widest case
takes the cluster-row kernels, whose partial rows are laid out per cluster),
a dx-only call must need no workspace at all, and a width too large for the
array must be refused.  This file is collected last so that a failure here
leaves every other test already run.
"""

import numpy as np
import pytest
import torch

import oracle as O
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
    lib = nl.load_library()
    # the set-up call the header asks for: N == 0 reserves nothing it needs later
    st = lib.ln_backward_static_workspace(None, 1, None, 1, None, None, None, None, 1, None, None, 0, 16, 1, 1,
                                          torch.cuda.current_stream().cuda_stream)
    assert st == 0


def _case(N, H, dt, seed):
    c = synth.norm_inputs(N, H, "bf16" if dt == torch.bfloat16 else "f32", seed=seed)
    return {k: v.to(DEV) for k, v in c.items()}


def _call(lib, t, mean, rstd, dx, dg, db, N, H, dt):
    return lib.ln_backward_static_workspace(
        t["dy"].data_ptr(), H, t["x"].data_ptr(), H, mean.data_ptr(), rstd.data_ptr(), t["gamma"].data_ptr(),
        dx.data_ptr(), H, None if dg is None else dg.data_ptr(), None if db is None else db.data_ptr(), N, H,
        CODE[dt], CODE[dt], torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("N,H,dt", [(2000, 1024, torch.bfloat16), (777, 5120, torch.bfloat16),
                                    (512, 16384, torch.bfloat16), (64, 256, torch.float32),
                                    (33, 1000, torch.bfloat16)])
def test_static_workspace_matches_oracle_and_ln_backward(N, H, dt):
    lib = nl.load_library()
    eps = 1e-5
    t = _case(N, H, dt, seed=N + H)
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"], eps)
    dx_ref, dg_ref, db_ref = nl.ln_backward(t["dy"], t["x"], mean, rstd, t["gamma"])
    torch.cuda.synchronize()
    x, dy, g = np64(t["x"]), np64(t["dy"]), np64(t["gamma"])
    dx_o, dg_o, db_o = O.layer_norm_backward(dy, x, g, eps)
    scale = ln_dx_scale(dy, x, g, eps)
    for call in range(2):  # the second call reuses the array the first one left behind
        dx = torch.empty_like(t["x"])
        dg = torch.empty(H, dtype=dt, device=DEV)
        db = torch.empty(H, dtype=dt, device=DEV)
        st = _call(lib, t, mean, rstd, dx, dg, db, N, H, dt)
        assert st == 0, nl._lib.status_str(st)
        torch.cuda.synchronize()
        check_out(np64(dx), dx_o, scale, dt, f"call {call} dx vs the oracle")
        check_param(np64(dg), dg_o, dt, f"call {call} dgamma vs the oracle")
        check_param(np64(db), db_o, dt, f"call {call} dbeta vs the oracle")
        check_out(np64(dx), np64(dx_ref), scale, dt, f"call {call} dx vs ln_backward")
        check_param(np64(dg), np64(dg_ref), dt, f"call {call} dgamma vs ln_backward")
        check_param(np64(db), np64(db_ref), dt, f"call {call} dbeta vs ln_backward")


def test_static_workspace_dx_only():
    """No parameter gradients: no partial rows, so any width is served."""
    lib = nl.load_library()
    N, H, dt, eps = 300, 2048, torch.bfloat16, 1e-5
    t = _case(N, H, dt, seed=5)
    y, mean, rstd = nl.ln_forward(t["x"], t["gamma"], t["beta"], eps)
    x, dy, g = np64(t["x"]), np64(t["dy"]), np64(t["gamma"])
    dx_o, _, _ = O.layer_norm_backward(dy, x, g, eps)
    for call in range(2):
        dx = torch.empty_like(t["x"])
        st = _call(lib, t, mean, rstd, dx, None, None, N, H, dt)
        assert st == 0, nl._lib.status_str(st)
        torch.cuda.synchronize()
        check_out(np64(dx), dx_o, ln_dx_scale(dy, x, g, eps), dt, f"call {call} dx only")


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
