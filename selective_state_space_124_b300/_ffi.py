"""ctypes declarations of include/ssm_scan.h (the C ABI of libssm_scan.so).

The library is loaded from this package directory only. There is no fallback: if it is missing the
import of the binding's entry points raises, naming the build command.
"""
from __future__ import annotations

import ctypes
import os

# the in-tree build's output (the same path build.py writes); build.py is not imported here, so that
# `python -m selective_state_space_124_b300.build` runs it as a fresh module
LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssm_scan.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT = range(5)
DTYPE = {"f32": 0, "bf16": 1}
DISC = {"euler": 0, "zoh": 1}

# Every symbol include/ssm_scan.h declares, with (restype, argtypes).
_vp, _i64, _i32, _fp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "ssm_scan_fwd": (_i32, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i64, _i64, _i64, _i64, _i32, _i32, _vp]),
    "ssm_scan_step": (_i32, [_fp, _vp, _vp, _fp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp]),
    "ssm_scan_fwd_host": (_i32, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _vp, ctypes.c_size_t, _i64, _i64, _i64, _i64,
                                 _i64, _i32, _i32, _vp]),
    "ssm_scan_fwd_host_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i32, _i64]),
    "ssm_scan_fwd_ex": (_i32, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _i32, _fp, _vp, _vp, _fp, _i64, _i64, _i64, _i64,
                               _i32, _i32, _vp]),
    "ssm_scan_step_ex": (_i32, [_fp, _vp, _vp, _fp, _vp, _vp, _fp, _i32, _fp, _vp, _vp, _i64, _i64, _i64, _i32, _i32,
                                _vp]),
    "ssm_scan_bwd": (_i32, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _vp, _vp, _fp, _fp, _fp, _fp, _vp, ctypes.c_size_t,
                            _i64, _i64, _i64, _i64, _i32, _i32, _vp]),
    "ssm_scan_bwd_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i64]),
    "ssm_scan_bwd_noalloc": (_i32, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _vp, _vp, _fp, _fp, _fp, _fp,
                                    _i64, _i64, _i64, _i64, _i32, _i32, _vp]),
    "ssm_ssd_fwd": (_i32, [_vp, _fp, _fp, _vp, _vp, _fp, _vp, _fp, _vp, ctypes.c_size_t, _i64, _i64, _i64, _i64, _i64,
                           _i32, _i32, _vp]),
    "ssm_ssd_fwd_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i64, _i64]),
    "ssm_check_device": (_i32, [_vp]),
    "ssm_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "ssm_status_string": (ctypes.c_char_p, [_i32]),
    "ssm_last_error": (ctypes.c_char_p, []),
    "ssm_version": (_i32, []),
}

_lib = None


class SsmError(RuntimeError):
    """A non-OK status from libssm_scan.so."""

    def __init__(self, func: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{func}: {status_name(status)}: {detail}")


def load(path: str = LIB) -> ctypes.CDLL:
    global _lib
    if _lib is not None and path == LIB:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m selective_state_space_124_b300.build` "
                           "(the CUDA library is required: there is no CPU path)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if path == LIB:
        _lib = lib
    return lib


def status_name(status: int) -> str:
    return load().ssm_status_string(status).decode()


def check(func: str, status: int) -> None:
    if status != SSM_OK:
        raise SsmError(func, status, load().ssm_last_error().decode())
