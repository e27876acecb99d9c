"""ctypes binding of libsinkattn's C ABI (include/sink_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. The library must be built (``attention_sink_softmax_gb300.build``);
if it is missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SINK_OK = 0
SINK_ERR_INVALID_ARG = 1
SINK_ERR_UNSUPPORTED = 2
SINK_ERR_CUDA = 3
SINK_ERR_WORKSPACE = 4
SINK_ERR_TIMEOUT = 5
SINK_ERR_DEVICE = 6
SINK_ERR_SCRATCH_LIMIT = 7

SINK_BF16 = 0
SINK_FP32 = 1

SINK_FLAG_TIMEOUT = 1
SINK_FLAG_SEQ_TOO_LONG = 2
SINK_FLAG_BAD_SEQLENS = 4

SINK_BWD_PREPARED = 1  # options bit of sink_attn_bwd_main_ex

# names declared in include/sink_attn.h, in declaration order
EXPORTS = (
    "sink_attn_workspace_bytes",
    "sink_attn_fwd",
    "sink_attn_fwd_ex",
    "sink_attn_bwd",
    "sink_attn_bwd_ex",
    "sink_attn_bwd_preprocess",
    "sink_attn_bwd_preprocess_ex",
    "sink_attn_bwd_main",
    "sink_attn_bwd_prepare",
    "sink_attn_bwd_main_ex",
    "sink_attn_fetch_device_error",
    "sink_attn_bwd_preprocess_noalloc",
    "sink_attn_noalloc_scratch_bytes",
    "sink_attn_decode_workspace_bytes",
    "sink_attn_decode",
    "sink_attn_status_str",
    "sink_attn_set_wait_limit_ns",
    "sink_attn_set_deterministic",
    "sink_attn_kernel_launches",
    "sink_attn_version",
)
# declared in include/sink_attn_testing.h
TESTING_EXPORTS = ("sink_attn_testing_withhold_load",)


class SinkAttnParams(ctypes.Structure):
    """Mirror of sink_attn_params_t."""
    _fields_ = [
        ("batch", ctypes.c_int),
        ("max_seqlen", ctypes.c_int),
        ("total_tokens", ctypes.c_int),
        ("h_q", ctypes.c_int),
        ("h_kv", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("causal", ctypes.c_int),
        ("window", ctypes.c_int),
    ]

    def __repr__(self):
        return "SinkAttnParams(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_PP = ctypes.POINTER(SinkAttnParams)


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libsinkattn (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libsinkattn is not built ({path} missing); run "
                    "attention_sink_softmax_gb300.build.build() or __graft_entry__.build()")
            L = ctypes.CDLL(path)
            L.sink_attn_workspace_bytes.argtypes = [_PP, ctypes.c_int]
            L.sink_attn_workspace_bytes.restype = ctypes.c_size_t
            L.sink_attn_fwd.argtypes = [_PP] + [_P] * 7 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_fwd.restype = ctypes.c_int
            L.sink_attn_fwd_ex.argtypes = [_PP] + [_P] * 8 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_fwd_ex.restype = ctypes.c_int
            L.sink_attn_bwd.argtypes = [_PP] + [_P] * 12 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_bwd.restype = ctypes.c_int
            L.sink_attn_bwd_ex.argtypes = [_PP] + [_P] * 13 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_bwd_ex.restype = ctypes.c_int
            L.sink_attn_bwd_preprocess.argtypes = [_PP] + [_P] * 6 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_bwd_preprocess.restype = ctypes.c_int
            L.sink_attn_bwd_preprocess_ex.argtypes = [_PP] + [_P] * 7 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_bwd_preprocess_ex.restype = ctypes.c_int
            L.sink_attn_bwd_main.argtypes = [_PP] + [_P] * 10 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_bwd_main.restype = ctypes.c_int
            L.sink_attn_bwd_prepare.argtypes = [_PP, _P, _P, _P, ctypes.c_size_t, _P]
            L.sink_attn_bwd_prepare.restype = ctypes.c_int
            L.sink_attn_bwd_main_ex.argtypes = ([_PP] + [_P] * 10 + [_P, ctypes.c_size_t, ctypes.c_uint, _P])
            L.sink_attn_bwd_main_ex.restype = ctypes.c_int
            L.sink_attn_fetch_device_error.argtypes = [_P, ctypes.c_size_t, _P,
                                                       ctypes.POINTER(ctypes.c_uint32)]
            L.sink_attn_fetch_device_error.restype = ctypes.c_int
            L.sink_attn_bwd_preprocess_noalloc.argtypes = [_PP] + [_P] * 6 + [_P]
            L.sink_attn_bwd_preprocess_noalloc.restype = ctypes.c_int
            L.sink_attn_noalloc_scratch_bytes.argtypes = []
            L.sink_attn_noalloc_scratch_bytes.restype = ctypes.c_size_t
            L.sink_attn_decode_workspace_bytes.argtypes = [_PP]
            L.sink_attn_decode_workspace_bytes.restype = ctypes.c_size_t
            L.sink_attn_decode.argtypes = [_PP] + [_P] * 8 + [_P, ctypes.c_size_t, _P]
            L.sink_attn_decode.restype = ctypes.c_int
            L.sink_attn_status_str.argtypes = [ctypes.c_int]
            L.sink_attn_status_str.restype = ctypes.c_char_p
            L.sink_attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.sink_attn_set_wait_limit_ns.restype = ctypes.c_uint64
            L.sink_attn_set_deterministic.argtypes = [ctypes.c_int]
            L.sink_attn_set_deterministic.restype = ctypes.c_int
            L.sink_attn_testing_withhold_load.argtypes = [ctypes.c_int]
            L.sink_attn_testing_withhold_load.restype = None
            L.sink_attn_kernel_launches.argtypes = []
            L.sink_attn_kernel_launches.restype = ctypes.c_uint64
            L.sink_attn_version.argtypes = []
            L.sink_attn_version.restype = ctypes.c_int
            _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().sink_attn_status_str(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != SINK_OK:
        raise SinkAttnError(status, where)
