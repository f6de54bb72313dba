"""ctypes view of libssm_scan.so, the library's C-ABI (include/ssm_scan.h).

The library must exist in-tree (built by ``python -m selective_state_space_155_b300.build``
or ``__graft_entry__.build()``); there is no fallback of any kind when it is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssm_scan.so")

SSM_OK = 0
SSM_ERR_NULL = -1
SSM_ERR_SHAPE = -2
SSM_ERR_DTYPE = -3
SSM_ERR_ALIGN = -4
SSM_ERR_UNSUPPORTED = -5
SSM_ERR_LAUNCH = -6
SSM_ERR_TIMEOUT = -7
SSM_ERR_ARG = -8

SSM_F32 = 0
SSM_BF16 = 1

SSM_DISC_DELTA_B = 0
SSM_DISC_ZOH = 1

SSM_FORM_PLAIN = 0
SSM_FORM_BALANCED = 1
SSM_FORM_SPLIT = 2
FORM_NAMES = {0: "plain", 1: "balanced", 2: "split"}

SSM_PROBE_EX2 = 0
SSM_PROBE_FFMA = 1
SSM_PROBE_FFMA2 = 2
SSM_PROBE_EX2_FFMA2 = 3
SSM_PROBE_RECURRENCE = 4
SSM_PROBE_WAIT_TIMEOUT = 5

# Every symbol the header declares, with its ctypes signature.
_vp, _fp, _i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "ssm_abi_version": (_i, []),
    "ssm_status_string": (ctypes.c_char_p, [_i]),
    "ssm_scan_fwd": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _vp, _fp, _i, _i, _i, _i, _i, _vp]),
    "ssm_scan_fwd_h0": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _fp, _i, _i, _i, _i, _i, _vp]),
    "ssm_scan_fwd_ex": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i, _vp]),
    "ssm_state_update": (_i, [_fp, _vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _vp, _i, _i, _i, _i, _vp]),
    "ssm_state_update_ex": (_i, [_fp, _vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _vp, _i, _i, _i, _i, _i, _vp]),
    "ssm_scan_num_checkpoints": (_i, [_i]),
    "ssm_scan_fwd_train": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _fp, _fp, _i, _i, _i, _i, _i,
                                _vp]),
    "ssm_scan_bwd": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _vp, _vp, _fp, _fp, _fp, _fp, _vp, _fp,
                          _fp, _i, _i, _i, _i, _i, _vp]),
    "ssm_scan_fwd_train_ex": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _fp, _fp, _i, _i, _i, _i, _i,
                                   _i, _vp]),
    "ssm_scan_bwd_ex": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _vp, _vp, _fp, _fp, _fp, _fp, _vp,
                             _fp, _fp, _i, _i, _i, _i, _i, _i, _vp]),
    "ssm_scan_fwd_form": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_int)]),
    "ssm_scan_fwd_ws": (_i, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _i, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i, _vp,
                             ctypes.c_size_t, _vp]),
    "ssm_scan_fwd_workspace_size": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]),
    "ssm_wait_timeouts": (_i, [ctypes.POINTER(ctypes.c_ulonglong)]),
    "ssm_probe_cycles": (_i, [_i, _vp, _i, _vp]),
    "ssm_probe_ops_per_cta": (ctypes.c_double, [_i]),
    "ssm_causal_conv1d_fwd": (_i, [_vp, _fp, _fp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "ssm_causal_conv1d_update": (_i, [_vp, _vp, _fp, _fp, _vp, _i, _i, _i, _i, _i, _vp]),
}

_lock = threading.Lock()
_lib = None


class SsmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library {LIB_PATH} is missing: build it with "
                                   "`python -m selective_state_space_155_b300.build`")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().ssm_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != SSM_OK:
        raise SsmError(fn, status)
