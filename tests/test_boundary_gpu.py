"""The Python binding refuses mis-shaped, mis-typed or misplaced arguments
before anything reaches the library: every bad argument below raises
ValueError, and the caller's output buffers keep their sentinel contents
(nothing was enqueued)."""

import pytest
import torch

import rmsnorm_ln_fwd_gb300 as nl
from rmsnorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu

N, H = 64, 256
SENTINEL = -7.25


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def t(dev):
    c = {k: v.to(dev) for k, v in synth.norm_inputs(N, H, "bf16", seed=11, with_residual=True,
                                                     with_dh_stream=True).items()}
    _, c["mean"], c["rstd"] = nl.ln_forward(c["x"], c["gamma"], c["beta"], 1e-5)
    torch.cuda.synchronize()
    return c


def _sentinel(shape, dev, dtype=torch.bfloat16):
    return torch.full(shape, SENTINEL, dtype=dtype, device=dev)


def _untouched(buf):
    torch.cuda.synchronize()
    return bool((buf.float() == SENTINEL).all())


def _bad_stats(t, dev):
    """(name, tensor) pairs that are not a contiguous fp32 CUDA vector of N."""
    return [("short", t["rstd"][: N - 1]),
            ("bf16", t["rstd"].to(torch.bfloat16)),
            ("host", t["rstd"].cpu()),
            ("strided", torch.zeros(2 * N, device=dev)[::2])]


def test_ln_backward_refuses(t, dev):
    x, dy, g = t["x"], t["dy"], t["gamma"]
    short = _sentinel((N - 1, H), dev)
    with pytest.raises(ValueError):
        nl.ln_backward(dy, x, t["mean"], t["rstd"], g, dx=short)
    assert _untouched(short)
    wrong_dtype = _sentinel((N, H), dev, torch.float32)
    with pytest.raises(ValueError):
        nl.ln_backward(dy, x, t["mean"], t["rstd"], g, dx=wrong_dtype)
    assert _untouched(wrong_dtype)
    for name, bad in _bad_stats(t, dev):
        out = _sentinel((N, H), dev)
        with pytest.raises(ValueError):
            nl.ln_backward(dy, x, bad, t["rstd"], g, dx=out)
        with pytest.raises(ValueError):
            nl.ln_backward(dy, x, t["mean"], bad, g, dx=out)
        assert _untouched(out), name
    out = _sentinel((N, H), dev)
    with pytest.raises(ValueError):
        nl.ln_backward(dy[:, : H // 2], x, t["mean"], t["rstd"], g, dx=out)   # dy narrower than x
    with pytest.raises(ValueError):
        nl.ln_backward(dy, x, t["mean"], t["rstd"], g.cpu(), dx=out)           # gamma on the host
    with pytest.raises(ValueError):
        nl.ln_backward(dy, x, t["mean"], t["rstd"], g, dx=out, workspace=torch.empty(1 << 20))  # host workspace
    assert _untouched(out)


def test_rms_backward_refuses(t, dev):
    x, dy, g = t["x"], t["dy"], t["gamma"]
    for name, bad in _bad_stats(t, dev):
        out = _sentinel((N, H), dev)
        with pytest.raises(ValueError):
            nl.rms_backward(dy, x, bad, g, dx=out)
        assert _untouched(out), name
    short = _sentinel((N - 2, H), dev)
    with pytest.raises(ValueError):
        nl.rms_backward(dy, x, t["rstd"], g, dx=short)
    assert _untouched(short)


def test_fused_backward_refuses(t, dev):
    h, dy, g = t["x"], t["dy"], t["gamma"]
    out = _sentinel((N, H), dev)
    for name, bad in _bad_stats(t, dev):
        with pytest.raises(ValueError):
            nl.fused_add_rms_backward(dy, h, bad, g, dx=out)
    with pytest.raises(ValueError):
        nl.fused_add_rms_backward(dy, h, t["rstd"], g, t["dh_stream"][: N - 1], dx=out)   # short stream gradient
    short = _sentinel((N - 1, H), dev)
    with pytest.raises(ValueError):
        nl.fused_add_rms_backward(dy, h, t["rstd"], g, dx=short)
    assert _untouched(out) and _untouched(short)


def test_from_output_backward_refuses(t, dev):
    y, dy, g, b = t["x"], t["dy"], t["gamma"], t["beta"]
    out = _sentinel((N, H), dev)
    for name, bad in _bad_stats(t, dev):
        with pytest.raises(ValueError):
            nl.ln_backward_from_output(dy, y, bad, g, b, dx=out)
        with pytest.raises(ValueError):
            nl.rms_backward_from_output(dy, y, bad, g, dx=out)
    short = _sentinel((N - 1, H), dev)
    with pytest.raises(ValueError):
        nl.ln_backward_from_output(dy, y, t["rstd"], g, b, dx=short)
    with pytest.raises(ValueError):
        nl.rms_backward_from_output(dy, y, t["rstd"], g, dx=short)
    with pytest.raises(ValueError):
        nl.ln_backward_from_output(dy, y, t["rstd"], g, b.cpu(), dx=out)
    assert _untouched(out) and _untouched(short)


def test_forwards_refuse(t, dev):
    x, r, g, b = t["x"], t["residual"], t["gamma"], t["beta"]
    short = _sentinel((N - 1, H), dev)
    with pytest.raises(ValueError):
        nl.ln_forward(x, g, b, out=short)
    with pytest.raises(ValueError):
        nl.rms_forward(x, g, out=short)
    with pytest.raises(ValueError):
        nl.fused_add_rms_forward(x, r, g, out=short)
    with pytest.raises(ValueError):
        nl.fused_add_rms_forward(x, r, g, h_out=short)
    with pytest.raises(ValueError):
        nl.fused_add_rms_forward(x, r[: N - 1], g)
    with pytest.raises(ValueError):
        nl.ln_forward(x, g.cpu(), b)
    with pytest.raises(ValueError):
        nl.ln_forward(x, g, b[: H - 1])
    assert _untouched(short)
