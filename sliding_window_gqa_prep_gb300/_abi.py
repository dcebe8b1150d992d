"""ctypes declarations of the C ABI in include/swa.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_float_p = ctypes.c_void_p   # device pointers travel as plain addresses

SWA_OK = 0
SWA_E_NULL = -1
SWA_E_SHAPE = -2
SWA_E_ALIGN = -3
SWA_E_WORKSPACE = -4
SWA_E_HAZARD = -5
SWA_E_CUDA = -6

SWA_DERR_META = 1
SWA_DERR_TIMEOUT = 2


class PrepArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("t", ctypes.c_int), ("nh", ctypes.c_int), ("nk", ctypes.c_int),
        ("hd", ctypes.c_int), ("cap", ctypes.c_int),
        ("eps", ctypes.c_float),
        ("yq", c_float_p), ("yk", c_float_p), ("yv", c_float_p), ("rope", c_float_p),
        ("q_scale", c_float_p), ("pos0", c_float_p),
        ("q_out", c_float_p), ("k_out", c_float_p), ("v_out", c_float_p),
        ("ring_k", c_float_p), ("ring_v", c_float_p),
        ("theta", ctypes.c_double),
    ]


class FarArgs(ctypes.Structure):
    _fields_ = [
        ("m", ctypes.c_int), ("rect", ctypes.c_int),
        ("k_tilde", ctypes.c_void_p), ("q_tilde", ctypes.c_void_p), ("mu", ctypes.c_void_p),
        ("mz", ctypes.c_void_p), ("t_hat", ctypes.c_void_p),
    ]


class AttendArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("t", ctypes.c_int), ("nh", ctypes.c_int), ("nk", ctypes.c_int),
        ("hd", ctypes.c_int), ("cap", ctypes.c_int), ("ns", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("meta", c_float_p), ("q", c_float_p), ("k_chunk", c_float_p), ("v_chunk", c_float_p),
        ("ring_k", c_float_p), ("ring_v", c_float_p), ("sink_k", c_float_p),
        ("sink_v", c_float_p), ("gate", c_float_p), ("gate_scale", c_float_p),
        ("out", c_float_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("commit", ctypes.c_int), ("meta_out", c_float_p), ("num_splits", ctypes.c_int),
        ("err", c_float_p), ("ev_start", ctypes.c_void_p), ("ev_stop", ctypes.c_void_p),
        ("far", ctypes.POINTER(FarArgs)), ("gate_ready", ctypes.c_void_p),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("nh", ctypes.c_int), ("nk", ctypes.c_int), ("hd", ctypes.c_int),
        ("cap", ctypes.c_int), ("ns", ctypes.c_int),
        ("scale", ctypes.c_float), ("eps", ctypes.c_float), ("theta", ctypes.c_double),
        ("yq", c_float_p), ("yk", c_float_p), ("yv", c_float_p), ("q_scale", c_float_p),
        ("pos0", c_float_p), ("meta", c_float_p),
        ("ring_k", c_float_p), ("ring_v", c_float_p), ("sink_k", c_float_p), ("sink_v", c_float_p),
        ("gate", c_float_p), ("gate_scale", c_float_p), ("out", c_float_p), ("meta_out", c_float_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("err", c_float_p), ("ev_start", ctypes.c_void_p), ("ev_stop", ctypes.c_void_p),
    ]


class FlashArgs(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int), ("nseg", ctypes.c_int), ("hd", ctypes.c_int), ("nh", ctypes.c_int),
        ("nk", ctypes.c_int),
        ("ld", ctypes.c_int), ("q_off", ctypes.c_int), ("k_off", ctypes.c_int), ("v_off", ctypes.c_int),
        ("ldo", ctypes.c_int), ("max_len", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("qkv", c_float_p), ("segs", ctypes.c_void_p), ("out", c_float_p), ("err", ctypes.c_void_p),
        ("ev_start", ctypes.c_void_p), ("ev_stop", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libswa_gb300.so (building it first if absent). Raises if it cannot
    be built or loaded: there is no fallback path."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if build_if_missing:
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with "
                           "python -m sliding_window_gqa_prep_gb300.build")
    lib = ctypes.CDLL(path)
    lib.swa_status_string.restype = ctypes.c_char_p
    lib.swa_status_string.argtypes = [ctypes.c_int]
    lib.swa_last_cuda_error.restype = ctypes.c_char_p
    lib.swa_last_cuda_error.argtypes = []
    lib.swa_version.restype = ctypes.c_char_p
    lib.swa_version.argtypes = []
    lib.swa_launch_count.restype = ctypes.c_uint64
    lib.swa_launch_count.argtypes = []
    lib.swa_rope_table.restype = ctypes.c_int
    lib.swa_rope_table.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
    lib.swa_prep.restype = ctypes.c_int
    lib.swa_prep.argtypes = [ctypes.POINTER(PrepArgs), ctypes.c_void_p]
    lib.swa_attend_workspace_size.restype = ctypes.c_size_t
    lib.swa_attend_workspace_size.argtypes = [ctypes.POINTER(AttendArgs)]
    lib.swa_attend_workspace_min.restype = ctypes.c_size_t
    lib.swa_attend_workspace_min.argtypes = [ctypes.POINTER(AttendArgs)]
    lib.swa_rollback.restype = ctypes.c_int
    lib.swa_rollback.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p]
    lib.swa_attend.restype = ctypes.c_int
    lib.swa_attend.argtypes = [ctypes.POINTER(AttendArgs), ctypes.c_void_p]
    lib.swa_attend_noalloc.restype = ctypes.c_int
    lib.swa_attend_noalloc.argtypes = [ctypes.POINTER(AttendArgs), ctypes.c_void_p]
    lib.swa_decode_step.restype = ctypes.c_int
    lib.swa_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.c_void_p]
    lib.swa_decode_workspace_size.restype = ctypes.c_size_t
    lib.swa_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs)]
    lib.swa_decode_launches.restype = ctypes.c_int
    lib.swa_decode_launches.argtypes = [ctypes.POINTER(DecodeArgs)]
    lib.swa_flash.restype = ctypes.c_int
    lib.swa_flash.argtypes = [ctypes.POINTER(FlashArgs), ctypes.c_void_p]
    lib.swa_flash_workspace_size.restype = ctypes.c_size_t
    lib.swa_flash_workspace_size.argtypes = [ctypes.POINTER(FlashArgs)]
    _lib = lib
    return lib


class SwaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load(build_if_missing=False)
        msg = lib.swa_status_string(status).decode()
        if status == SWA_E_CUDA:
            msg += " (" + lib.swa_last_cuda_error().decode() + ")"
        super().__init__(f"{where}: status {status}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != SWA_OK:
        raise SwaError(status, where)
