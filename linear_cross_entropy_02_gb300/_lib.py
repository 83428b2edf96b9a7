"""ctypes declarations of the C ABI in include/flce.h (libflce.so, built in-tree)."""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libflce.so")

FLCE_OK = 0
FLCE_ERR_ARG = 1
FLCE_ERR_ALIGN = 2
FLCE_ERR_WORKSPACE = 3
FLCE_ERR_UNSUPPORTED = 4
FLCE_ERR_CUDA = 5
FLCE_ERR_LABEL = 16
FLCE_ERR_TIMEOUT = 32
FLCE_ERR_NONFINITE = 64

FLCE_MODE_CE_ONLY = 0
FLCE_MODE_FORWARD = 1
FLCE_MODE_FORWARD_BACKWARD = 2
FLCE_MODE_CROSS_ENTROPY = 3
FLCE_MODE_FORWARD_BACKWARD_HOST = 4
FLCE_MODE_CE_ONLY_HOST = 5

FLCE_REDUCTION_MEAN = 0
FLCE_REDUCTION_SUM = 1
FLCE_REDUCTION_NONE = 2

FLCE_DTYPE_BF16 = 0
FLCE_DTYPE_F32 = 1

FLCE_FLAG_SIMT_GEMM = 1
FLCE_FLAG_TEST_STALL = 2
FLCE_FLAG_KMAJOR_BWD = 4
FLCE_FLAG_RECOMPUTE = 8
FLCE_FLAG_TILE128 = 16
FLCE_FLAG_TILE256 = 32
FLCE_FLAG_CTA_PAIR = 64
FLCE_FLAG_F32_3PASS = 128
FLCE_FLAG_VP_STORED = 256

FLCE_NUM_KERNELS = 17

EXPORTED = [
    "flce_default_params", "flce_workspace_size", "flce_chunk_rows", "flce_ce_only", "flce_ce_only_noalloc", "flce_forward",
    "flce_forward_backward", "flce_forward_backward_from_host", "flce_ce_only_from_host", "flce_cross_entropy",
    "flce_scale_gradient", "flce_get_status", "flce_status_string", "flce_launch_count", "flce_profile_begin",
    "flce_profile_read", "flce_kernel_name", "flce_vp_workspace_size", "flce_vp_forward", "flce_vp_backward",
]


class FlceParams(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int64),
        ("hidden", ctypes.c_int64),
        ("vocab", ctypes.c_int64),
        ("ld_h", ctypes.c_int64),
        ("ld_w", ctypes.c_int64),
        ("softcap", ctypes.c_float),
        ("out_mult", ctypes.c_float),
        ("ignore_index", ctypes.c_int64),
        ("reduction", ctypes.c_int32),
        ("grad_scale", ctypes.c_float),
        ("chunk_rows", ctypes.c_int64),
        ("flags", ctypes.c_int32),
        ("timeout_ns", ctypes.c_int64),
        ("vocab_slab", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
    ]


class FlceError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({status_string(code)})")
        self.code = code


_lib = None
_lock = threading.Lock()

_P = ctypes.POINTER(FlceParams)
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded libflce.so. Raises if the library has not been built: there
    is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(nvcc, sm_103a). There is no CPU or PyTorch fallback.")
        L = ctypes.CDLL(LIB_PATH)
        L.flce_default_params.argtypes = [_P]
        L.flce_default_params.restype = None
        L.flce_workspace_size.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.flce_workspace_size.restype = _sz
        L.flce_chunk_rows.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.flce_chunk_rows.restype = ctypes.c_int64
        L.flce_ce_only.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.flce_ce_only.restype = ctypes.c_int
        L.flce_ce_only_noalloc.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.flce_ce_only_noalloc.restype = ctypes.c_int
        L.flce_forward.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.flce_forward.restype = ctypes.c_int
        L.flce_forward_backward.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.flce_forward_backward.restype = ctypes.c_int
        L.flce_cross_entropy.argtypes = [_P, _vp, ctypes.c_int, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _sz, _vp]
        L.flce_cross_entropy.restype = ctypes.c_int
        L.flce_forward_backward_from_host.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                                      _vp]
        L.flce_forward_backward_from_host.restype = ctypes.c_int
        L.flce_ce_only_from_host.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]
        L.flce_ce_only_from_host.restype = ctypes.c_int
        L.flce_scale_gradient.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int64, _vp, _vp]
        L.flce_scale_gradient.restype = ctypes.c_int
        L.flce_get_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]
        L.flce_get_status.restype = ctypes.c_int
        L.flce_status_string.argtypes = [ctypes.c_int]
        L.flce_status_string.restype = ctypes.c_char_p
        L.flce_launch_count.argtypes = []
        L.flce_launch_count.restype = ctypes.c_int64
        L.flce_profile_begin.argtypes = [ctypes.c_int]
        L.flce_profile_begin.restype = ctypes.c_int
        L.flce_profile_read.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                                        ctypes.c_int]
        L.flce_profile_read.restype = ctypes.c_int
        L.flce_kernel_name.argtypes = [ctypes.c_int]
        L.flce_kernel_name.restype = ctypes.c_char_p
        L.flce_vp_workspace_size.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.flce_vp_workspace_size.restype = _sz
        L.flce_vp_forward.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.flce_vp_forward.restype = ctypes.c_int
        L.flce_vp_backward.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int64), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _vp, _vp, _sz, _vp]
        L.flce_vp_backward.restype = ctypes.c_int
        _lib = L
        return L


def status_string(code: int) -> str:
    try:
        return lib().flce_status_string(int(code)).decode()
    except Exception:  # the library may be what failed to load
        return "unknown"
