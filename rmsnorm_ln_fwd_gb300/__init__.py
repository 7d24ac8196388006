"""Row-wise LayerNorm and RMSNorm for one GB300 GPU (sm_103a).

Forward, fused residual-add + RMSNorm forward, and the training backward, all
computed by the hand-written CUDA kernels of ``libnorm.so`` behind the C ABI in
``include/norm.h``.  This package only marshals arguments to that library;
there is no CPU or PyTorch fallback.
"""

from ._lib import NormError, load as load_library, LIB_PATH  # noqa: F401
from .ops import (  # noqa: F401
    bwd_workspace_bytes,
    fused_add_rms_backward,
    fused_add_rms_forward,
    ln_backward,
    ln_backward_from_output,
    ln_forward,
    rms_backward,
    rms_backward_from_output,
    rms_forward,
)

__all__ = [
    "ln_forward",
    "rms_forward",
    "fused_add_rms_forward",
    "fused_add_rms_backward",
    "ln_backward",
    "rms_backward",
    "ln_backward_from_output",
    "rms_backward_from_output",
    "bwd_workspace_bytes",
    "NormError",
    "load_library",
]
