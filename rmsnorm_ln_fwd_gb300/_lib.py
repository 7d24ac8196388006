"""ctypes loader for libnorm.so, the C ABI declared in include/norm.h.

The library must have been built (``rmsnorm_ln_fwd_gb300._build.build()``);
there is no fallback of any kind.  A missing or unloadable library raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnorm.so")

NORM_OK = 0
NORM_ERR_INVALID_VALUE = 1
NORM_ERR_UNSUPPORTED = 2
NORM_ERR_WORKSPACE = 3
NORM_ERR_CUDA = 4

NORM_F32 = 0
NORM_BF16 = 1
NORM_F16 = 2

# name -> (restype, argtypes), one entry per function declared in include/norm.h
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_I = ctypes.c_int
SIGNATURES = {
    "ln_forward": (_I, [_P, _I64, _P, _P, _P, _I64, _P, _P, _I64, _I64, _F, _I, _I, _P]),
    "rms_forward": (_I, [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _I, _I, _P]),
    "fused_add_rms_forward": (_I, [_P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _P, _I64, _I64, _F, _I, _I, _P]),
    "norm_bwd_workspace_bytes": (ctypes.c_size_t, [_I64, _I]),
    "ln_backward": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _P, _P, ctypes.c_size_t, _I64, _I64,
                         _I, _I, _P]),
    "rms_backward": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _P, ctypes.c_size_t, _I64, _I64, _I, _I, _P]),
    "ln_backward_from_output": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _P, _P, ctypes.c_size_t, _I64,
                                     _I64, _I, _I, _P]),
    "rms_backward_from_output": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _P, ctypes.c_size_t, _I64, _I64,
                                      _I, _I, _P]),
    "fused_add_rms_backward": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _I64, _P, _P,
                                    ctypes.c_size_t, _I64, _I64, _I, _I, _P]),
    "ln_backward_static_workspace": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _P, _I64, _I64, _I, _I,
                                         _P]),
    "norm_status_str": (ctypes.c_char_p, [_I]),
    "norm_abi_version": (_I, []),
    "norm_last_error": (ctypes.c_char_p, []),
    "norm_device_errors": (_I, [_I, ctypes.POINTER(ctypes.c_uint), _I]),
    "norm_selftest_bounded_wait": (_I, [ctypes.c_ulonglong, _P]),
    "norm_set_kernel_path": (_I, [_I]),
    "norm_set_bwd_split_event": (_I, [_P]),
}

_lock = threading.Lock()
_lib = None


class NormError(RuntimeError):
    """A libnorm entry point returned a status other than NORM_OK."""

    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libnorm.so once and declare every signature; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libnorm.so not found at {LIB_PATH}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_str(status: int) -> str:
    return load().norm_status_str(int(status)).decode()


def device_errors(device: int = 0, clear: bool = True) -> int:
    """Error bits the kernels raised on `device` since the last clear."""
    v = ctypes.c_uint(0)
    check("norm_device_errors", load().norm_device_errors(int(device), ctypes.byref(v), int(clear)))
    return int(v.value)


def set_kernel_path(path: int) -> None:
    """0: automatic (default), 1: register rows, 2: strided loop, 3: bulk-copy pipeline first."""
    check("norm_set_kernel_path", load().norm_set_kernel_path(int(path)))


def set_bwd_split_event(event_handle) -> None:
    """Record the raw cudaEvent_t `event_handle` (an int, or None to stop)
    between every later backward's main kernel and its partial reduction."""
    check("norm_set_bwd_split_event", load().norm_set_bwd_split_event(event_handle or None))


def check(fn: str, status: int) -> None:
    if status != NORM_OK:
        text = status_str(status)
        if status == NORM_ERR_CUDA:
            text += f" [{load().norm_last_error().decode()}]"
        raise NormError(fn, status, text)
