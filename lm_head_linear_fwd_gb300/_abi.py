"""ctypes binding of libflce.so (argument marshalling only).

Every function here has the name and argument order of the C entry point in
``include/flce.h`` / ``include/flce_gemm.h``.  Nothing here computes: the work
runs in the library's kernels.  If the library is missing the import fails
loudly; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import platform

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", platform.machine(), "libflce.so")

FLCE_OK = 0
FLCE_ELABEL = -5
FLCE_ETIMEOUT = -9
FLCE_EBOUNDS = -10
FLCE_BF16 = 0
FLCE_F32 = 1
FLCE_SUM = 0
FLCE_MEAN = 1

_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_p = ctypes.c_void_p

_SIGNATURES = {
    "flce_status_string": (ctypes.c_char_p, [_i]),
    "flce_last_cuda_error": (ctypes.c_char_p, []),
    "ce_logits_workspace_bytes": (_sz, [_i64, _i64]),
    "ce_logits_fwd": (_i, [_p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _p, _p,
                           _p, _sz, _p, _p]),
    "ce_logits_fwd_noalloc": (_i, [_p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _p,
                                   _p]),
    "ce_logits_bwd": (_i, [_p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _i, _p,
                           _i64, _p, _p]),
    "ce_logits_fwd_bwd_workspace_bytes": (_sz, [_i64, _i64]),
    "ce_logits_fwd_bwd": (_i, [_p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _p, _i,
                               _p, _i64, _p, _sz, _p, _p]),
    "flce_workspace_bytes": (_sz, [_i, _i64, _i64, _i64, _i64]),
    "flce_default_chunk": (_i64, [_i, _i64, _i64, _i64]),
    "flce_fwd": (_i, [_p, _p, _p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _p, _p,
                      _p, _sz, _p, _p]),
    "flce_bwd": (_i, [_p, _p, _p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p, _p, _i64,
                      _p, _p, _i, _p, _p, _sz, _p, _p]),
    "flce_fwd_shard": (_i, [_p, _p, _p, _i, _i64, _i64, _i64, _i64, _i64, _p, _i64, _p, _p, _p,
                            _p, _sz, _p, _p]),
    "flce_shard_rescale": (_i, [_p, _p, _p, _i64, _p, _p]),
    "flce_shard_finish": (_i, [_p, _p, _p, _p, _i64, _i64, _i64, _i, _i64, _p, _p, _p, _p, _p,
                               _sz, _p, _p]),
    "flce_bwd_shard": (_i, [_p, _p, _p, _i, _i64, _i64, _i64, _i64, _i64, _p, _i64, _i, _i64, _p,
                            _p, _p, _i64, _p, _p, _i, _p, _p, _sz, _p, _p]),
    "ce_logits_fwd_shard": (_i, [_p, _i, _i64, _i64, _i64, _i64, _i64, _p, _i64, _p, _p, _p, _p,
                                 _p]),
    "ce_logits_bwd_shard": (_i, [_p, _i, _i64, _i64, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _p,
                                 _p, _i, _p, _i64, _p, _p]),
    "flce_fwd_bwd_workspace_bytes": (_sz, [_i, _i64, _i64, _i64, _i64]),
    "flce_fwd_bwd": (_i, [_p, _p, _p, _i, _i64, _i64, _i64, _p, _i64, _i, _i64, _p, _i64, _p, _p,
                          _p, _p, _p, _p, _i, _p, _p, _sz, _p, _p]),
    "flce_grad_scale": (_i, [_p, _i, _i64, _p, _p]),
    "flce_count_valid": (_i, [_p, _i64, _i64, _i64, _p, _p]),
    "flce_wait_selftest": (_i, [_p, ctypes.c_uint64, _p]),
    "flce_device_checks": (_i, []),
    "flce_bounds_selftest": (_i, [_p, _p]),
    "flce_mask_packed_labels": (_i, [_p, _p, _i64, _i64, _i64, _p]),
    "flce_gemm_set_pair": (_i, [_i]),
    "flce_gemm_pair_slots": (_i, []),
    "flce_gemm": (_i, [_i, _i, _i, _i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _i, _p, _p]),
}

EXPORTED = tuple(_SIGNATURES)

_lib = None


def open_library(path: str) -> ctypes.CDLL:
    """Opens a build of the library at `path` with every signature set (the
    package itself always uses libflce.so through load())."""
    if not os.path.exists(path):
        raise ImportError(
            f"libflce.so not found at {path}: build it with "
            "`python lm_head_linear_fwd_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libflce.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = open_library(path)
    return _lib


def status_string(code: int) -> str:
    return load().flce_status_string(int(code)).decode()


class FlceError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = f"{where}: {status_string(code)} ({code})"
        if self.code == -7:
            msg += " [" + load().flce_last_cuda_error().decode() + "]"
        super().__init__(msg)


def check(rc: int, where: str) -> None:
    if rc != FLCE_OK:
        raise FlceError(rc, where)


def _call(name):
    def f(*args):
        return getattr(load(), name)(*args)
    f.__name__ = name
    return f


flce_status_string = _call("flce_status_string")
flce_last_cuda_error = _call("flce_last_cuda_error")
ce_logits_workspace_bytes = _call("ce_logits_workspace_bytes")
ce_logits_fwd = _call("ce_logits_fwd")
ce_logits_fwd_noalloc = _call("ce_logits_fwd_noalloc")
ce_logits_bwd = _call("ce_logits_bwd")
ce_logits_fwd_bwd_workspace_bytes = _call("ce_logits_fwd_bwd_workspace_bytes")
ce_logits_fwd_bwd = _call("ce_logits_fwd_bwd")
flce_workspace_bytes = _call("flce_workspace_bytes")
flce_default_chunk = _call("flce_default_chunk")
flce_fwd = _call("flce_fwd")
flce_bwd = _call("flce_bwd")
flce_gemm = _call("flce_gemm")
flce_fwd_bwd_workspace_bytes = _call("flce_fwd_bwd_workspace_bytes")
flce_fwd_shard = _call("flce_fwd_shard")
flce_shard_rescale = _call("flce_shard_rescale")
flce_shard_finish = _call("flce_shard_finish")
flce_bwd_shard = _call("flce_bwd_shard")
ce_logits_fwd_shard = _call("ce_logits_fwd_shard")
ce_logits_bwd_shard = _call("ce_logits_bwd_shard")
flce_fwd_bwd = _call("flce_fwd_bwd")
flce_grad_scale = _call("flce_grad_scale")
flce_count_valid = _call("flce_count_valid")
flce_wait_selftest = _call("flce_wait_selftest")
flce_device_checks = _call("flce_device_checks")
flce_bounds_selftest = _call("flce_bounds_selftest")
flce_mask_packed_labels = _call("flce_mask_packed_labels")
flce_gemm_set_pair = _call("flce_gemm_set_pair")
flce_gemm_pair_slots = _call("flce_gemm_pair_slots")
