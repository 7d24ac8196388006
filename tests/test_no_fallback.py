"""The binding has no CPU path: host tensors are refused before any call, and
a missing libnorm.so is an error, never a silent fallback (CPU, no GPU)."""

import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import rmsnorm_ln_fwd_gb300 as nl  # noqa: E402
from rmsnorm_ln_fwd_gb300 import _lib  # noqa: E402

N, H = 4, 64


def _host():
    g = torch.Generator().manual_seed(0)
    t = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    rs = torch.ones(N, dtype=torch.float32)
    return t(N, H), t(N, H), t(H), t(H), rs


CALLS = {
    "ln_forward": lambda x, dy, g, b, rs: nl.ln_forward(x, g, b),
    "rms_forward": lambda x, dy, g, b, rs: nl.rms_forward(x, g),
    "fused_add_rms_forward": lambda x, dy, g, b, rs: nl.fused_add_rms_forward(x, dy, g),
    "ln_backward": lambda x, dy, g, b, rs: nl.ln_backward(dy, x, rs, rs, g),
    "rms_backward": lambda x, dy, g, b, rs: nl.rms_backward(dy, x, rs, g),
    "fused_add_rms_backward": lambda x, dy, g, b, rs: nl.fused_add_rms_backward(dy, x, rs, g),
    "ln_backward_from_output": lambda x, dy, g, b, rs: nl.ln_backward_from_output(dy, x, rs, g, b),
    "rms_backward_from_output": lambda x, dy, g, b, rs: nl.rms_backward_from_output(dy, x, rs, g),
}


def test_every_op_is_covered():
    ops = {n for n in nl.__all__ if n.endswith(("_forward", "_backward", "_from_output"))}
    assert ops == set(CALLS)


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name](*_host())


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libnorm.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()
