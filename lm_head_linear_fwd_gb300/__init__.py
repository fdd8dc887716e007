"""Language-model loss head for GB300 (sm_103a): cross-entropy on given logits
and fused linear cross-entropy, as hand-written CUDA kernels behind a C ABI
(``include/flce.h``), with a thin PyTorch binding.

Importing the package loads ``_lib/libflce.so``; it raises if the library has
not been built (``python lm_head_linear_fwd_gb300/build.py``).
"""
from . import _abi

_abi.load()

from .api import (  # noqa: E402,F401
    BackwardOut, ForwardOut, ce_logits, ce_logits_bwd, ce_logits_fwd, ce_logits_fwd_bwd,
    ce_logits_fwd_bwd_workspace_bytes, ce_logits_workspace_bytes, check_status, flce, flce_bwd, flce_default_chunk, flce_fwd,
    flce_fwd_bwd, flce_gemm, flce_workspace_bytes, grad_scale_, mask_packed_labels, new_status,
)
from ._abi import FlceError  # noqa: E402,F401
