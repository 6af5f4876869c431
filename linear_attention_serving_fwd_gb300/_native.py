"""ctypes binding of ``libkda.so`` (include/kda.h).  Argument marshalling only.

The shared library is built in-tree by :mod:`.build`.  Loading fails loudly
if it cannot be built or loaded: there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None
_variant = None  # None: the regular library; "phase_timing": the measurement build

KDA_OK = 0
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_UNSUPPORTED_DTYPE = 2
KDA_ERR_CUDA = 3
KDA_ERR_DEVICE_TIMEOUT = 4
KDA_ERR_DEVICE_INDEX = 5
KDA_ERR_DEVICE_RANGE = 6
KDA_DTYPE_BF16 = 0
KDA_DTYPE_FP16 = 1

# Every symbol include/kda.h declares.
EXPORTS = ("kda_chunk_workspace_bytes", "kda_chunk_fwd", "kda_decode", "kda_verify",
           "kda_last_error", "kda_last_error_message", "kda_device_status", "kda_trace_enable", "kda_trace_read",
           "kda_version", "kda_chunk_fwd_noalloc", "kda_commit", "kda_chunk_fwd_ex",
           "kda_decode_steps", "kda_verify_ex", "kda_commit_ex", "kda_chunk_fwd_host",
           "kda_chunk_fwd_host_workspace_bytes", "kda_conv_scratch_bytes", "kda_selftest_wait_timeout")


class KdaActivations(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_stride_tok", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("k", ctypes.c_void_p), ("k_stride_tok", ctypes.c_int64), ("k_stride_head", ctypes.c_int64),
        ("v", ctypes.c_void_p), ("v_stride_tok", ctypes.c_int64), ("v_stride_head", ctypes.c_int64),
        ("g", ctypes.c_void_p), ("g_stride_tok", ctypes.c_int64), ("g_stride_head", ctypes.c_int64),
        ("beta", ctypes.c_void_p), ("beta_stride_tok", ctypes.c_int64),
        ("beta_stride_head", ctypes.c_int64),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("dtype", ctypes.c_int32), ("t_total", ctypes.c_int32),
        ("hqk", ctypes.c_int32), ("hv", ctypes.c_int32),
        ("use_qk_l2norm", ctypes.c_int32),
        ("scale", ctypes.c_float), ("lower_bound", ctypes.c_float),
        ("state_bf16", ctypes.c_int32),
    ]


class KdaConv(ctypes.Structure):
    _fields_ = [
        ("weight", ctypes.c_void_p), ("weight_f32", ctypes.c_int32),
        ("state", ctypes.c_void_p),
        ("row_stride", ctypes.c_int64), ("pos_stride", ctypes.c_int64),
        ("chan_stride", ctypes.c_int64), ("rows", ctypes.c_int64),
        ("positions", ctypes.c_int32),
        ("state_indices", ctypes.c_void_p), ("has_initial_state", ctypes.c_void_p),
        ("num_accepted", ctypes.c_void_p),
        ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t),
    ]


class KdaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[kda status {code}] {msg}")
        self.code = code


def _declare(lib):
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    A = ctypes.POINTER(KdaActivations)
    lib.kda_chunk_workspace_bytes.argtypes = [I32, I32, I32, I32]
    lib.kda_chunk_workspace_bytes.restype = SZ
    lib.kda_chunk_fwd.argtypes = [A, P, P, I32, P, P, P, I64, I64, P, P, I32, P, SZ, P]
    lib.kda_chunk_fwd.restype = ctypes.c_int
    CV = ctypes.POINTER(KdaConv)
    lib.kda_chunk_fwd_ex.argtypes = [A, P, P, I32, P, P, P, I64, I64, P, P, P, I64, I64, P, P, CV, I32, P,
                                     SZ, P]
    lib.kda_chunk_fwd_ex.restype = ctypes.c_int
    lib.kda_chunk_fwd_noalloc.argtypes = [A, P, P, I32, P, P, P, I64, I64, P, P, I32, P]
    lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
    lib.kda_chunk_fwd_host.argtypes = [A, P, P, I32, P, P, I32, I32, P, SZ, P]
    lib.kda_chunk_fwd_host.restype = ctypes.c_int
    lib.kda_chunk_fwd_host_workspace_bytes.argtypes = [A, P, I32, I32, I32]
    lib.kda_chunk_fwd_host_workspace_bytes.restype = SZ
    lib.kda_conv_scratch_bytes.argtypes = [I32, I32, I32]
    lib.kda_conv_scratch_bytes.restype = SZ
    lib.kda_decode.argtypes = [A, P, P, I64, I64, P, P, I32, I32, P]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_decode_steps.argtypes = [A, P, P, I64, I64, P, P, I64, P, I32, I32, P]
    lib.kda_decode_steps.restype = ctypes.c_int
    lib.kda_verify.argtypes = [A, P, P, I64, I64, P, P, I32, I32, P, P, P, P]
    lib.kda_verify.restype = ctypes.c_int
    lib.kda_verify_ex.argtypes = [A, P, P, I64, I64, P, P, I32, I32, P, P, P, CV, P]
    lib.kda_verify_ex.restype = ctypes.c_int
    lib.kda_commit.argtypes = [P, I64, I64, P, P, I32, I32, I32, P, P, P, P, ctypes.c_float, P]
    lib.kda_commit.restype = ctypes.c_int
    lib.kda_commit_ex.argtypes = [P, I64, I64, P, P, I32, I32, I32, P, P, P, P, ctypes.c_float, I32, I32, P]
    lib.kda_commit_ex.restype = ctypes.c_int
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_last_error_message.argtypes = []
    lib.kda_last_error_message.restype = ctypes.c_char_p
    lib.kda_device_status.argtypes = [P, I32]
    lib.kda_device_status.restype = ctypes.c_int
    lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.kda_selftest_wait_timeout.restype = ctypes.c_int
    lib.kda_trace_enable.argtypes = [I32]
    lib.kda_trace_enable.restype = ctypes.c_int
    lib.kda_trace_read.argtypes = [I32, ctypes.c_char_p, I32, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(I32)]
    lib.kda_trace_read.restype = ctypes.c_int
    lib.kda_version.argtypes = []
    lib.kda_version.restype = ctypes.c_char_p
    return lib


def lib_path() -> str:
    return _build.lib_path(_variant)


def select_variant(name) -> None:
    """Load a measurement build (``"phase_timing"``) instead of the regular
    library; only before the library is first used in this process."""
    global _variant
    with _lock:
        if _lib is not None:
            raise RuntimeError("select_variant must come before the library is loaded")
        _variant = name


def lib():
    """The loaded library (built in-tree on first use if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build(variant=_variant)
            if not os.path.exists(path):
                raise ImportError(f"libkda.so missing at {path}")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def check(rc: int):
    if rc == KDA_OK:
        return
    msg = lib().kda_last_error_message().decode()
    if rc == KDA_ERR_INVALID_ARGUMENT:
        raise ValueError(msg)
    if rc == KDA_ERR_UNSUPPORTED_DTYPE:
        raise TypeError(msg)
    raise KdaError(rc, msg)


def trace_enable(on: bool):
    lib().kda_trace_enable(1 if on else 0)


def trace_read() -> dict:
    """{kernel name: (total ms, launches)} recorded since trace_enable(True)."""
    L = lib()
    n = L.kda_trace_read(-1, None, 0, None, None)
    out = {}
    for i in range(n):
        buf = ctypes.create_string_buffer(128)
        ms = ctypes.c_double()
        cnt = ctypes.c_int32()
        L.kda_trace_read(i, buf, 128, ctypes.byref(ms), ctypes.byref(cnt))
        out[buf.value.decode()] = (ms.value, cnt.value)
    return out
