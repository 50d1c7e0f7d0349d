"""ctypes view of the C ABI in include/attn_gb300.h (argument marshalling only).

Loads ``libattn_gb300.so`` from this package directory.  Nothing here computes any part
of attention: every step runs in the library's CUDA kernels.  If the library is missing
the import of the binding fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn_gb300.so")

ATTN_DTYPE_BF16 = 1
ATTN_DTYPE_F32 = 2

ATTN_SOFTMAX_DEFAULT = 0
ATTN_SOFTMAX_OFF_BY_ONE = 1

ATTN_OK = 0
ATTN_ERR_INVALID = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_WORKSPACE = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_DEVICE = 5

# Every function the header declares (tests check the library exports each one).
EXPORTS = (
    "attn_fwd_workspace_size", "attn_fwd", "attn_bwd_workspace_size", "attn_bwd",
    "attn_check_device_status", "attn_status_string", "attn_path_name", "attn_launch_counter",
    "attn_profile_next_main_kernel", "attn_profile_next_aux_kernels", "attn_fwd_noalloc", "attn_noalloc_check_device_status",
    "attn_selftest_wait_expiry", "attn_meta_size", "attn_meta_build",
)


class AttnArgs(ctypes.Structure):
    """Mirror of ``attn_args``."""
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("B", ctypes.c_int), ("Sq", ctypes.c_int), ("Sk", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("q", ctypes.c_void_p),
        ("q_stride_b", ctypes.c_int64), ("q_stride_s", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
        ("k", ctypes.c_void_p),
        ("k_stride_b", ctypes.c_int64), ("k_stride_s", ctypes.c_int64), ("k_stride_h", ctypes.c_int64),
        ("v", ctypes.c_void_p),
        ("v_stride_b", ctypes.c_int64), ("v_stride_s", ctypes.c_int64), ("v_stride_h", ctypes.c_int64),
        ("bias", ctypes.c_void_p),
        ("bias_stride_b", ctypes.c_int64), ("bias_stride_h", ctypes.c_int64),
        ("seg_q", ctypes.c_void_p), ("seg_k", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("nseq", ctypes.c_int),
        ("causal", ctypes.c_int), ("window", ctypes.c_int),
        ("softcap", ctypes.c_float), ("sink", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("softmax_type", ctypes.c_int), ("kv_splits", ctypes.c_int),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("meta", ctypes.c_void_p),
    ]


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with attention_flash_attn_gb300.build.build() "
                "(the CUDA library is the only implementation; there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        A = ctypes.POINTER(AttnArgs)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        L.attn_fwd_workspace_size.argtypes = [A]
        L.attn_fwd_workspace_size.restype = sz
        L.attn_bwd_workspace_size.argtypes = [A]
        L.attn_bwd_workspace_size.restype = sz
        L.attn_meta_size.argtypes = [A]
        L.attn_meta_size.restype = sz
        L.attn_meta_build.argtypes = [A, vp, sz, vp]
        L.attn_meta_build.restype = ctypes.c_int
        L.attn_fwd.argtypes = [A, vp, vp, vp, sz, vp]
        L.attn_fwd.restype = ctypes.c_int
        L.attn_fwd_noalloc.argtypes = [A, vp, vp, vp]
        L.attn_fwd_noalloc.restype = ctypes.c_int
        L.attn_noalloc_check_device_status.argtypes = [vp]
        L.attn_noalloc_check_device_status.restype = ctypes.c_int
        L.attn_selftest_wait_expiry.argtypes = [vp, sz, ctypes.c_uint64, vp]
        L.attn_selftest_wait_expiry.restype = ctypes.c_int
        L.attn_bwd.argtypes = [A, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_bwd.restype = ctypes.c_int
        L.attn_check_device_status.argtypes = [vp, vp]
        L.attn_check_device_status.restype = ctypes.c_int
        L.attn_status_string.argtypes = [ctypes.c_int]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_path_name.argtypes = [A]
        L.attn_path_name.restype = ctypes.c_char_p
        L.attn_profile_next_main_kernel.argtypes = [vp, vp]
        L.attn_profile_next_main_kernel.restype = None
        L.attn_profile_next_aux_kernels.argtypes = [vp, vp, vp, vp]
        L.attn_profile_next_aux_kernels.restype = None
        L.attn_launch_counter.argtypes = []
        L.attn_launch_counter.restype = ctypes.c_uint64
        _lib = L
    return _lib


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib().attn_status_string(status).decode()} (status {status})")
