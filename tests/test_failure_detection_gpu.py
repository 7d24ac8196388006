"""Failure detection on the GPU without a GPU fault.

Every wait inside the kernels is bounded and reports through the per-device
error word instead of trapping.  Here a self-test kernel waits (50 ms limit)
on a barrier that nothing ever signals: the wait must run out, the host must
read NORM_DEVICE_ERR_WAIT_TIMEOUT, and the context must stay usable for a
normal call afterwards.
"""

import pytest
import torch

import oracle as O
import rmsnorm_ln_fwd_gb300 as nl
from normtest import check_bf16, ln_y_scale, np64
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    nl.load_library()


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = nl.load_library()
    torch.cuda.synchronize()
    nl._lib.device_errors(0, clear=True)
    st = lib.norm_selftest_bounded_wait(50_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()  # returns: the wait gave up instead of hanging
    assert nl._lib.device_errors(0, clear=True) & 1
    assert nl._lib.device_errors(0, clear=True) == 0  # cleared
    # the context still works: a normal call, checked against the oracle
    c = {k: v.cuda() for k, v in synth.norm_inputs(16, 1024, "bf16", seed=9).items()}
    y, mean, rstd = nl.ln_forward(c["x"], c["gamma"], c["beta"])
    torch.cuda.synchronize()
    x, g, b = np64(c["x"]), np64(c["gamma"]), np64(c["beta"])
    yr, mr, rr = O.layer_norm_forward(x, g, b, 1e-5)
    check_bf16(np64(y), yr, ln_y_scale(x, mr, rr, g, b), "y after the self-test")
    assert nl._lib.device_errors(0, clear=True) == 0
