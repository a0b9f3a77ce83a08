"""ctypes view of libssmscan's C ABI (include/ssmscan.h): structs, enums, signatures.

Loading never falls back to anything: if the shared library is missing it is built
with nvcc (see build.py), and if that fails the error propagates.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SSM_OK = 0
SSM_ERR_INVALID_ARG = 1
SSM_ERR_UNSUPPORTED = 2
SSM_ERR_CUDA = 3
SSM_ERR_TIMEOUT = 4

SSM_F32 = 0
SSM_BF16 = 1

SSM_DISC_EXP_EULER = 0
SSM_DISC_ZOH = 1

SSM_SCAN_KERNEL_AUTO = 0
SSM_SCAN_KERNEL_TMEM = 1
SSM_SCAN_KERNEL_TMA = 2
SSM_SCAN_KERNEL_TILED = 3
SSM_SCAN_KERNEL_GENERIC = 4

ABI_VERSION = 2

_vp = ctypes.c_void_p
_fp = ctypes.c_void_p  # float* passed as an address
_i = ctypes.c_int


class ScanParams(ctypes.Structure):
    _fields_ = [("batch", _i), ("dim", _i), ("dstate", _i), ("seqlen", _i), ("ngroups", _i),
                ("in_dtype", _i), ("out_dtype", _i),
                ("x", _vp), ("delta", _vp), ("delta_bias", _fp), ("delta_softplus", _i),
                ("A", _fp), ("B", _vp), ("C", _vp), ("D_skip", _fp), ("z", _vp), ("h0", _fp),
                ("y", _vp), ("h_final", _fp), ("disc", _i)]


class ScanOpts(ctypes.Structure):
    _fields_ = [("kernel", _i), ("threads_per_channel", _i), ("max_segments", _i),
                ("wait_limit", ctypes.c_uint), ("fault_test", _i)]


class ScanBwdParams(ctypes.Structure):
    _fields_ = [("fwd", ScanParams), ("dy", _vp), ("dh_final", _fp), ("dx", _fp),
                ("ddelta", _fp), ("dz", _fp), ("dA", _fp), ("dB", _fp), ("dC", _fp),
                ("dD_skip", _fp), ("ddelta_bias", _fp), ("dh0", _fp)]


class Mamba3Params(ctypes.Structure):
    _fields_ = [("batch", _i), ("dim", _i), ("dstate", _i), ("seqlen", _i), ("ngroups", _i),
                ("in_dtype", _i), ("out_dtype", _i),
                ("x", _vp), ("delta", _vp), ("delta_bias", _fp), ("delta_softplus", _i),
                ("A_re", _fp), ("A_im", _fp), ("lam", _vp), ("B", _vp), ("C", _vp),
                ("D_skip", _fp), ("z", _vp), ("h0", _fp), ("y", _vp), ("h_final", _fp)]


class S4dParams(ctypes.Structure):
    _fields_ = [("batch", _i), ("dim", _i), ("dstate", _i), ("seqlen", _i), ("in_dtype", _i),
                ("out_dtype", _i), ("u", _vp), ("log_dt", _fp), ("A", _fp), ("B", _fp),
                ("C", _fp), ("D_skip", _fp), ("h0", _fp), ("y", _vp), ("h_final", _fp)]


class SsdParams(ctypes.Structure):
    _fields_ = [("batch", _i), ("seqlen", _i), ("nheads", _i), ("headdim", _i), ("dstate", _i),
                ("ngroups", _i), ("chunk_size", _i), ("in_dtype", _i), ("out_dtype", _i),
                ("x", _vp), ("dt", _vp), ("dt_bias", _fp), ("dt_softplus", _i), ("A", _fp),
                ("B", _vp), ("C", _vp), ("D_skip", _fp), ("z", _vp), ("h0", _fp), ("y", _vp),
                ("h_final", _fp), ("disc", _i)]


class SsdBwdParams(ctypes.Structure):
    _fields_ = [("fwd", SsdParams), ("dy", _vp), ("dh_final", _fp), ("dx", _fp), ("ddt", _fp),
                ("dz", _fp), ("dA", _fp), ("dB", _fp), ("dC", _fp), ("dD_skip", _fp),
                ("ddt_bias", _fp), ("dh0", _fp)]


class StepParams(ctypes.Structure):
    _fields_ = [("batch", _i), ("nheads", _i), ("headdim", _i), ("dstate", _i), ("ngroups", _i),
                ("a_per_state", _i), ("in_dtype", _i), ("out_dtype", _i),
                ("state", _fp), ("x", _vp), ("dt", _vp), ("dt_bias", _fp), ("dt_softplus", _i),
                ("A", _fp), ("B", _vp), ("C", _vp), ("D_skip", _fp), ("z", _vp), ("y", _vp),
                ("disc", _i)]


SYMBOLS = ("ssm_scan_fwd", "ssm_scan_fwd_ex", "ssm_scan_workspace_size", "ssm_scan_bwd",
           "ssm_scan_bwd_workspace_size", "ssm_mamba3_scan_fwd", "ssm_mamba3_scan_workspace_size", "ssm_s4d_scan_fwd",
           "ssm_s4d_scan_workspace_size", "ssm_s4d_conv_fwd", "ssm_s4d_conv_workspace_size",
           "ssm_s4d_kernel", "ssd_scan_bwd", "ssd_scan_bwd_workspace_size", "ssd_chunk_scan_fwd",
           "ssd_chunk_scan_workspace_size", "ssm_state_update", "ssm_state_update_tokens",
           "ssm_last_error", "ssm_abi_version", "ssm_device_status", "ssm_wait_timeouts")

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """The loaded libssmscan (built first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libssmscan not found at {_build.LIB}")
            lib = ctypes.CDLL(_build.LIB)
            sz = ctypes.c_size_t
            lib.ssm_scan_fwd.restype = _i
            lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanParams), _vp]
            lib.ssm_scan_fwd_ex.restype = _i
            lib.ssm_scan_fwd_ex.argtypes = [ctypes.POINTER(ScanParams), ctypes.POINTER(ScanOpts),
                                            _vp, sz, _vp]
            lib.ssm_scan_workspace_size.restype = sz
            lib.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanParams),
                                                    ctypes.POINTER(ScanOpts)]
            lib.ssm_scan_bwd.restype = _i
            lib.ssm_scan_bwd.argtypes = [ctypes.POINTER(ScanBwdParams), _vp, sz, _vp]
            lib.ssm_scan_bwd_workspace_size.restype = sz
            lib.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(ScanBwdParams)]
            lib.ssm_mamba3_scan_fwd.restype = _i
            lib.ssm_mamba3_scan_fwd.argtypes = [ctypes.POINTER(Mamba3Params), _vp, sz, _vp]
            lib.ssm_mamba3_scan_workspace_size.restype = sz
            lib.ssm_mamba3_scan_workspace_size.argtypes = [ctypes.POINTER(Mamba3Params)]
            lib.ssm_s4d_scan_fwd.restype = _i
            lib.ssm_s4d_scan_fwd.argtypes = [ctypes.POINTER(S4dParams), _vp, sz, _vp]
            lib.ssm_s4d_scan_workspace_size.restype = sz
            lib.ssm_s4d_scan_workspace_size.argtypes = [ctypes.POINTER(S4dParams)]
            lib.ssm_s4d_conv_fwd.restype = _i
            lib.ssm_s4d_conv_fwd.argtypes = [ctypes.POINTER(S4dParams), _vp, sz, _vp]
            lib.ssm_s4d_conv_workspace_size.restype = sz
            lib.ssm_s4d_conv_workspace_size.argtypes = [ctypes.POINTER(S4dParams)]
            lib.ssm_s4d_kernel.restype = _i
            lib.ssm_s4d_kernel.argtypes = [ctypes.POINTER(S4dParams), _vp, _i, _vp]
            lib.ssd_scan_bwd.restype = _i
            lib.ssd_scan_bwd.argtypes = [ctypes.POINTER(SsdBwdParams), _vp, sz, _vp]
            lib.ssd_scan_bwd_workspace_size.restype = sz
            lib.ssd_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(SsdBwdParams)]
            lib.ssd_chunk_scan_fwd.restype = _i
            lib.ssd_chunk_scan_fwd.argtypes = [ctypes.POINTER(SsdParams), _vp, sz, _vp]
            lib.ssd_chunk_scan_workspace_size.restype = sz
            lib.ssd_chunk_scan_workspace_size.argtypes = [ctypes.POINTER(SsdParams)]
            lib.ssm_state_update.restype = _i
            lib.ssm_state_update.argtypes = [ctypes.POINTER(StepParams), _vp]
            lib.ssm_state_update_tokens.restype = _i
            lib.ssm_state_update_tokens.argtypes = [ctypes.POINTER(StepParams), _i, _vp]
            lib.ssm_last_error.restype = ctypes.c_char_p
            lib.ssm_last_error.argtypes = []
            lib.ssm_abi_version.restype = _i
            lib.ssm_abi_version.argtypes = []
            lib.ssm_wait_timeouts.restype = ctypes.c_uint
            lib.ssm_wait_timeouts.argtypes = []
            lib.ssm_device_status.restype = _i
            lib.ssm_device_status.argtypes = []
            if lib.ssm_abi_version() != ABI_VERSION:
                raise RuntimeError(f"libssmscan ABI version {lib.ssm_abi_version()}, this "
                                   f"binding expects {ABI_VERSION}: rebuild the library")
            _lib = lib
        return _lib


class SsmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status
        self.message = message


def check(status: int):
    if status != SSM_OK:
        msg = load(False).ssm_last_error().decode(errors="replace")
        raise SsmError(status, msg)
