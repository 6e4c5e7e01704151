"""ctypes loader for libfa.so: the C ABI of include/fa.h, nothing more."""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_SCRATCH_LIMIT = 5
FA_ERR_DEVICE_ARG = 6
NOALLOC_SCRATCH_BYTES = 8 << 20

FA_BF16 = 0
FA_FP16 = 1

FA_OFFSET_BOTTOM_RIGHT = -(1 << 63)

# Every function the header declares (checked against include/fa.h by the tests).
EXPORTS = (
    "fa_fwd",
    "fa_num_splits_heuristic",
    "fa_splitkv_default_splits",
    "fa_splitkv_workspace_size",
    "fa_fwd_splitkv",
    "fa_fwd_splitkv_noalloc",
    "fa_kvcache_workspace_size",
    "fa_fwd_kvcache",
    "fa_fwd_varlen",
    "fa_bwd_workspace_size",
    "fa_bwd",
    "fa_quantize_e4m3",
    "fa_splitkv_e4m3_workspace_size",
    "fa_fwd_splitkv_e4m3",
    "fa_fwd_e4m3",
    "fa_splitkv_combine",
    "fa_sync_status",
    "fa_selftest_wait_timeout",
    "fa_status_string",
    "fa_version",
)


class FwdArgs(ctypes.Structure):
    """Mirror of `fa_fwd_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("sq", ctypes.c_int32),
        ("skv", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 3),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("o_strides", ctypes.c_int64 * 3),
        ("causal", ctypes.c_int32),
        ("q_pos_offset", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("local", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("softcap", ctypes.c_float),
    ]


class KvcacheArgs(ctypes.Structure):
    """Mirror of `fa_kvcache_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 2),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int32),
        ("seqlens_k", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("max_seqlen_k", ctypes.c_int32),
        ("o", ctypes.c_void_p),
        ("o_strides", ctypes.c_int64 * 2),
        ("lse", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("local", ctypes.c_int32),
        ("window_left", ctypes.c_int32),
        ("softcap", ctypes.c_float),
    ]


class VarlenArgs(ctypes.Structure):
    """Mirror of `fa_varlen_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
        ("total_k", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 2),
        ("k_strides", ctypes.c_int64 * 2),
        ("v_strides", ctypes.c_int64 * 2),
        ("o_strides", ctypes.c_int64 * 2),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("causal", ctypes.c_int32),
        ("local", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
    ]


class BwdArgs(ctypes.Structure):
    """Mirror of `fa_bwd_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("sq", ctypes.c_int32),
        ("skv", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("dout", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 3),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("o_strides", ctypes.c_int64 * 3),
        ("do_strides", ctypes.c_int64 * 3),
        ("dq_strides", ctypes.c_int64 * 3),
        ("dk_strides", ctypes.c_int64 * 3),
        ("dv_strides", ctypes.c_int64 * 3),
        ("causal", ctypes.c_int32),
        ("q_pos_offset", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("local", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("softcap", ctypes.c_float),
    ]


class QuantArgs(ctypes.Structure):
    """Mirror of `fa_quant_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("s", ctypes.c_int32),
        ("h", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("x_strides", ctypes.c_int64 * 3),
        ("out", ctypes.c_void_p),
        ("out_strides", ctypes.c_int64 * 3),
        ("transpose", ctypes.c_int32),
        ("per_head", ctypes.c_int32),
        ("descale", ctypes.c_void_p),
    ]


class E4m3Args(ctypes.Structure):
    """Mirror of `fa_fwd_e4m3_args`."""

    _fields_ = [
        ("b", ctypes.c_int32),
        ("sq", ctypes.c_int32),
        ("skv", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("vt", ctypes.c_void_p),
        ("q_descale", ctypes.c_void_p),
        ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 3),
        ("k_strides", ctypes.c_int64 * 3),
        ("vt_strides", ctypes.c_int64 * 3),
        ("o_strides", ctypes.c_int64 * 3),
        ("causal", ctypes.c_int32),
        ("q_pos_offset", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("local", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
    ]


class SplitkvE4m3Args(ctypes.Structure):
    """Mirror of `fa_splitkv_e4m3_args`."""

    _fields_ = [
        ("dtype", ctypes.c_int),
        ("b", ctypes.c_int32),
        ("skv", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("q_strides", ctypes.c_int64 * 2),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("o_strides", ctypes.c_int64 * 2),
        ("lse", ctypes.c_void_p),
        ("scale", ctypes.c_float),
    ]


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load():
    """Load libfa.so; raise if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run `python -m tiled_exact_attention_gb300.build`)")
        lib = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        pargs = ctypes.POINTER(FwdArgs)
        lib.fa_fwd.argtypes = [pargs, vp]
        lib.fa_fwd.restype = ctypes.c_int
        lib.fa_num_splits_heuristic.argtypes = [i64, i64, i64, i32]
        lib.fa_num_splits_heuristic.restype = i32
        lib.fa_splitkv_default_splits.argtypes = [pargs]
        lib.fa_splitkv_default_splits.restype = i32
        lib.fa_splitkv_workspace_size.argtypes = [pargs, i32]
        lib.fa_splitkv_workspace_size.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv.argtypes = [pargs, i32, vp, ctypes.c_size_t, ctypes.POINTER(i32), vp]
        lib.fa_fwd_splitkv.restype = ctypes.c_int
        lib.fa_fwd_splitkv_noalloc.argtypes = [pargs, i32, ctypes.POINTER(i32), vp]
        lib.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
        pkv = ctypes.POINTER(KvcacheArgs)
        lib.fa_kvcache_workspace_size.argtypes = [pkv, i32]
        lib.fa_kvcache_workspace_size.restype = ctypes.c_size_t
        lib.fa_fwd_kvcache.argtypes = [pkv, i32, vp, ctypes.c_size_t, ctypes.POINTER(i32), vp]
        lib.fa_fwd_kvcache.restype = ctypes.c_int
        lib.fa_fwd_varlen.argtypes = [ctypes.POINTER(VarlenArgs), vp]
        lib.fa_fwd_varlen.restype = ctypes.c_int
        lib.fa_bwd_workspace_size.argtypes = [ctypes.POINTER(BwdArgs)]
        lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
        lib.fa_bwd.argtypes = [ctypes.POINTER(BwdArgs), vp, ctypes.c_size_t, vp]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_quantize_e4m3.argtypes = [ctypes.POINTER(QuantArgs), vp]
        lib.fa_quantize_e4m3.restype = ctypes.c_int
        lib.fa_fwd_e4m3.argtypes = [ctypes.POINTER(E4m3Args), vp]
        lib.fa_fwd_e4m3.restype = ctypes.c_int
        pse = ctypes.POINTER(SplitkvE4m3Args)
        lib.fa_splitkv_e4m3_workspace_size.argtypes = [pse, i32]
        lib.fa_splitkv_e4m3_workspace_size.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv_e4m3.argtypes = [pse, i32, vp, ctypes.c_size_t, ctypes.POINTER(i32), vp]
        lib.fa_fwd_splitkv_e4m3.restype = ctypes.c_int
        lib.fa_splitkv_combine.argtypes = [vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, vp,
                                           ctypes.POINTER(i64), vp, vp]
        lib.fa_splitkv_combine.restype = ctypes.c_int
        lib.fa_sync_status.argtypes = [vp]
        lib.fa_sync_status.restype = ctypes.c_int
        lib.fa_selftest_wait_timeout.argtypes = [vp]
        lib.fa_selftest_wait_timeout.restype = ctypes.c_int
        lib.fa_status_string.argtypes = [ctypes.c_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except Exception:  # the library itself may be what is missing
        return "status"


def check(status: int, what: str) -> None:
    if status != FA_OK:
        raise FaError(status, what)
