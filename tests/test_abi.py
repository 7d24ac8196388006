"""The C-ABI library on the CPU: it builds, loads, exports every function the
header declares, and validates arguments on the host before any CUDA call.

Pointers passed here are fake addresses; validation never dereferences them
and every call below is rejected (or has N == 0) before reaching the GPU.
"""

import os
import re
import shutil
import subprocess

import pytest
import torch

from rmsnorm_ln_fwd_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "norm.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA = 0, 1, 2, 3, 4
F32, BF16 = 0, 1
A, B, C, D = 0x100000, 0x200000, 0x300000, 0x400000  # fake, well-separated addresses


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:norm_status|size_t|const char\*|int)\s+([a-z_0-9]+)\s*\(", text, flags=re.M)


def test_header_declares_the_five_ops():
    names = set(declared_functions())
    for op in ["ln_forward", "rms_forward", "fused_add_rms_forward", "ln_backward", "rms_backward",
               "fused_add_rms_backward", "ln_backward_from_output", "rms_backward_from_output",
               "norm_bwd_workspace_bytes", "norm_status_str"]:
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported by libnorm.so"
        assert n in _lib.SIGNATURES, f"{n} has no binding"
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
        exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
        assert set(names) <= exported


def test_header_is_plain_c():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    p = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert p.returncode == 0, p.stderr


def test_status_strings_and_version(lib):
    for code in range(5):
        s = lib.norm_status_str(code).decode()
        assert s.startswith("NORM_")
    assert lib.norm_status_str(99).decode() == "NORM_ERR_UNKNOWN"
    assert lib.norm_abi_version() == 10000


def _ln(lib, **kw):
    a = dict(x=A, ldx=64, g=None, b=None, y=B, ldy=64, mean=None, rstd=None, N=4, H=64, eps=1e-5, xd=BF16,
             wd=BF16)
    a.update(kw)
    return lib.ln_forward(a["x"], a["ldx"], a["g"], a["b"], a["y"], a["ldy"], a["mean"], a["rstd"], a["N"],
                          a["H"], a["eps"], a["xd"], a["wd"], None)


def test_forward_validation(lib):
    assert _ln(lib, xd=F32, wd=BF16) == UNSUPPORTED
    assert _ln(lib, xd=7) == UNSUPPORTED
    for eps in (0.0, -1e-5, float("nan"), float("inf")):
        assert _ln(lib, eps=eps) == INVALID
    assert _ln(lib, H=0) == INVALID
    assert _ln(lib, N=-1) == INVALID
    assert _ln(lib, H=(1 << 24) + 1, ldx=(1 << 24) + 1, ldy=(1 << 24) + 1) == INVALID
    assert _ln(lib, ldx=63) == INVALID
    assert _ln(lib, x=None) == INVALID
    assert _ln(lib, y=A + 2) == INVALID            # y partially overlaps x
    assert _ln(lib, y=A, ldy=65) == INVALID        # same start, different stride
    assert _ln(lib, mean=C, rstd=C + 4) == INVALID  # mean/rstd overlap
    assert _ln(lib, N=0, x=None, y=None) == OK      # nothing to do
    assert lib.rms_forward(A, 64, None, B, 64, None, 4, 64, -1.0, BF16, BF16, None) == INVALID


def test_fused_validation(lib):
    def f(x=A, r=B, y=C, h=D, ld=64, N=4, H=64, ldh=64):
        return lib.fused_add_rms_forward(x, ld, r, ld, None, y, ld, h, ldh, None, N, H, 1e-6, BF16, BF16, None)
    assert f(h=None) == INVALID
    assert f(r=None) == INVALID
    assert f(y=A) == INVALID              # y may not alias an input
    assert f(y=D) == INVALID              # nor h
    assert f(h=A + 64) == INVALID         # h partially overlaps x
    assert f(h=B, ldh=65) == INVALID      # h over residual with another stride
    assert f(r=A + 8, h=A) == INVALID     # in place over x while residual overlaps x
    assert f(N=0, x=None, r=None, y=None, h=None) == OK


def test_forward_stats_and_params_clear_of_outputs(lib):
    # mean/rstd (outputs) and gamma/beta (inputs) may not overlap each other,
    # the output rows or (for the statistics) the input rows
    E = 0x600000
    assert _ln(lib, g=B) == INVALID                          # gamma under y
    assert _ln(lib, b=B + 64) == INVALID                     # beta under y
    assert _ln(lib, mean=A + 8) == INVALID                   # mean over x
    assert _ln(lib, rstd=B + 8) == INVALID                   # rstd over y
    assert _ln(lib, g=E, mean=E + 8) == INVALID              # mean over gamma
    assert _ln(lib, b=E, rstd=E) == INVALID                  # rstd over beta
    assert lib.fused_add_rms_forward(A, 64, B, 64, D + 8, C, 64, D, 64, None, 4, 64, 1e-6, BF16, BF16,
                                     None) == INVALID      # gamma under h
    assert lib.fused_add_rms_forward(A, 64, B, 64, None, C, 64, D, 64, B + 4, 4, 64, 1e-6, BF16, BF16,
                                     None) == INVALID      # rstd over the residual
    assert lib.rms_forward(A, 64, B + 2, B, 64, None, 4, 64, 1e-5, BF16, BF16, None) == INVALID  # gamma under y


def test_backward_stats_and_params_clear_of_outputs(lib):
    E, F = 0x600000, 0x700000
    assert _bwd(lib, mean=D + 16) == INVALID                 # mean under dx
    assert _bwd(lib, rstd=D) == INVALID                      # rstd under dx
    assert _bwd(lib, g=D + 32) == INVALID                    # gamma under dx
    assert _bwd(lib, g=E, dg=E + 2, ws=F, wsb=1 << 20) == INVALID  # dgamma over gamma
    assert _bwd(lib, dg=B + 2, ws=F, wsb=1 << 20) == INVALID  # dgamma over x
    assert _bwd(lib, db=A, ws=F, wsb=1 << 20) == INVALID     # dbeta over dy
    assert _bwd(lib, dg=C + 4, ws=F, wsb=1 << 20) == INVALID  # dgamma over mean
    assert _bwd(lib, dg=E, ws=B - 16, wsb=64) == WORKSPACE   # workspace over x
    assert _bwd(lib, dg=E, ws=C, wsb=64) == WORKSPACE        # workspace over mean
    assert _bwd(lib, dg=E, ws=D + 64, wsb=64) == WORKSPACE   # workspace over dx
    assert _bwd(lib, dg=E, ws=None) == WORKSPACE
    assert _bwd(lib, dg=E, ws=F + 4, wsb=64) == WORKSPACE    # misaligned workspace


def _bwd(lib, **kw):
    a = dict(dy=A, ldy=64, x=B, ldx=64, mean=C, rstd=C + 4096, g=None, dx=D, lddx=64, dg=None, db=None, ws=None,
             wsb=0, N=4, H=64, xd=BF16, wd=BF16)
    a.update(kw)
    return lib.ln_backward(a["dy"], a["ldy"], a["x"], a["ldx"], a["mean"], a["rstd"], a["g"], a["dx"], a["lddx"],
                           a["dg"], a["db"], a["ws"], a["wsb"], a["N"], a["H"], a["xd"], a["wd"], None)


def test_backward_validation(lib):
    assert _bwd(lib, xd=BF16, wd=7) == UNSUPPORTED
    assert _bwd(lib, rstd=None) == INVALID
    assert _bwd(lib, mean=None) == INVALID
    assert _bwd(lib, dx=B) == INVALID            # dx may not overlap x
    assert _bwd(lib, dx=A + 2) == INVALID        # partial overlap with dy
    assert _bwd(lib, H=0) == INVALID
    assert _bwd(lib, lddx=10) == INVALID
    assert _bwd(lib, dg=0x500000, db=0x500000 + 8) == INVALID  # dgamma/dbeta overlap
    assert lib.rms_backward(A, 64, B, 64, None, None, D, 64, None, None, 0, 4, 64, BF16, BF16, None) == INVALID


def _fbwd(lib, **kw):
    a = dict(dy=A, lddy=64, h=B, ldh=64, rstd=C, g=None, dh=None, lddh=0, dx=D, lddx=64, dres=None, lddres=0,
             dg=None, ws=None, wsb=0, N=4, H=64, xd=BF16, wd=BF16)
    a.update(kw)
    return lib.fused_add_rms_backward(a["dy"], a["lddy"], a["h"], a["ldh"], a["rstd"], a["g"], a["dh"], a["lddh"],
                                      a["dx"], a["lddx"], a["dres"], a["lddres"], a["dg"], a["ws"], a["wsb"], a["N"],
                                      a["H"], a["xd"], a["wd"], None)


def test_fused_backward_validation(lib):
    assert _fbwd(lib, wd=7) == UNSUPPORTED
    assert _fbwd(lib, rstd=None) == INVALID
    assert _fbwd(lib, h=None) == INVALID
    assert _fbwd(lib, dx=B) == INVALID                      # dx over h
    assert _fbwd(lib, dx=A + 2) == INVALID                  # dx partly over dy
    assert _fbwd(lib, dh=0x500000, lddh=10) == INVALID      # short stream-gradient stride
    assert _fbwd(lib, dh=D + 2, lddh=64) == INVALID         # stream gradient partly under dx
    assert _fbwd(lib, dres=B, lddres=64) == INVALID         # dres over h
    assert _fbwd(lib, dres=D + 2, lddres=64) == INVALID     # dres partly over dx
    assert _fbwd(lib, dres=D, lddres=72) == INVALID         # dres at dx with another stride
    assert _fbwd(lib, dres=A + 2, lddres=64) == INVALID     # dres partly over dy
    assert _fbwd(lib, dres=0x500000, lddres=10) == INVALID  # short dres stride
    assert _fbwd(lib, dh=0x500000, lddh=64, dres=0x500000 + 2, lddres=64) == INVALID  # dres partly over dh


def test_fused_backward_clear_of_outputs(lib):
    E = 0x600000
    assert _fbwd(lib, rstd=0x500000, dres=0x500000 - 64, lddres=64) == INVALID       # rstd under dres
    assert _fbwd(lib, dg=0x500000 + 8, dres=0x500000, lddres=64, ws=E, wsb=1 << 20) == INVALID  # dgamma under dres
    assert _fbwd(lib, dg=0x500000 + 8, dh=0x500000, lddh=64, ws=E, wsb=1 << 20) == INVALID  # dgamma over dh_in
    assert _fbwd(lib, g=D + 8) == INVALID                                              # gamma under dx


def test_from_output_validation(lib):
    def ln(**kw):
        a = dict(dy=A, lddy=64, y=B, ldy=64, rstd=C, g=None, b=None, dx=D, lddx=64, dg=None, db=None, ws=None,
                 wsb=0, N=4, H=64, xd=BF16, wd=BF16)
        a.update(kw)
        return lib.ln_backward_from_output(a["dy"], a["lddy"], a["y"], a["ldy"], a["rstd"], a["g"], a["b"], a["dx"],
                                           a["lddx"], a["dg"], a["db"], a["ws"], a["wsb"], a["N"], a["H"], a["xd"],
                                           a["wd"], None)
    assert ln(wd=9) == UNSUPPORTED
    assert ln(xd=F32, wd=BF16) == UNSUPPORTED
    assert ln(rstd=None) == INVALID
    assert ln(y=None) == INVALID
    assert ln(dx=B) == INVALID          # dx over y
    assert ln(dx=A + 2) == INVALID      # dx partly over dy
    assert ln(ldy=10) == INVALID
    assert ln(H=0) == INVALID
    assert ln(dg=0x500000, db=0x500000 + 4) == INVALID
    assert ln(b=D + 4) == INVALID       # beta under dx
    assert lib.rms_backward_from_output(A, 64, B, 64, None, None, D, 64, None, None, 0, 4, 64, BF16, BF16,
                                        None) == INVALID
    assert lib.rms_backward_from_output(A, 64, B, 64, C, None, B + 8, 64, None, None, 0, 4, 64, BF16, BF16,
                                        None) == INVALID


def test_selftest_limit_validation(lib):
    assert lib.norm_selftest_bounded_wait(10, None) == INVALID          # below 1 ms
    assert lib.norm_selftest_bounded_wait(3_000_000_000, None) == INVALID  # above 2 s


def test_kernel_path_override_validation(lib):
    assert lib.norm_set_kernel_path(4) == INVALID
    assert lib.norm_set_kernel_path(-1) == INVALID
    for p in (3, 2, 1, 0):
        assert lib.norm_set_kernel_path(p) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_reports_cuda_error(lib):
    # valid arguments, but no GPU to run on: a clean NORM_ERR_CUDA, no crash
    assert _ln(lib) == CUDA
    assert lib.norm_bwd_workspace_bytes(1024, 0) == 0
    assert lib.norm_bwd_workspace_bytes(0, 0) == 0
