"""ctypes declarations of the C ABI in include/ers.h (argument marshalling only).

Loading fails loudly when libers.so is missing or lacks a symbol: there is no CPU or
PyTorch fallback for any operation of this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libers.so")

ERS_OK = 0
STATUS_NAMES = {
    0: "ERS_OK", 1: "ERS_EINVAL", 2: "ERS_ESHAPE", 3: "ERS_EDTYPE", 4: "ERS_EPTR", 5: "ERS_EALIGN",
    6: "ERS_EOVERFLOW", 7: "ERS_ECOMMIT", 8: "ERS_ESLOT", 9: "ERS_ETIMEOUT", 10: "ERS_EWORKSPACE",
    11: "ERS_ECUDA", 12: "ERS_EUNSUPPORTED",
}
DTYPE_F32 = 0
DTYPE_BF16 = 1
FLAG_FUSE_REFRESH = 1
FLAG_REPLAYSSM = 2
FLAG_AUTO_FLUSH = 4

READ_BF16 = 0
READ_FP8_E4M3 = 1
READ_NVFP4 = 2

ANCHOR_F32 = 0
ANCHOR_F16_SR = 1
ANCHOR_NVFP4_SHARED_SR = 2

# Every function include/ers.h declares.
EXPORTS = (
    "ers_status_str", "ers_version", "ers_ssd_scan_fwd_workspace_size", "ers_ssd_scan_fwd",
    "ers_chunked_prefill_workspace_size", "ers_chunked_prefill", "ers_replay_decode", "ers_refresh",
    "ers_spec_verify", "ers_commit", "ers_ssu_update", "ers_ssd_scan_fwd_static", "ers_conv1d_fwd",
    "ers_conv1d_update", "ers_gdn_verify", "ers_gdn_commit", "ers_gdn_refresh", "ers_selftest_bounded_wait",
    "ers_spec_verify_exact_workspace_size", "ers_spec_verify_exact", "ers_commit_exact",
)


class ErsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_str(code)})")


class Dims(ctypes.Structure):
    _fields_ = [("nheads", ctypes.c_int32), ("ngroups", ctypes.c_int32), ("headdim", ctypes.c_int32),
                ("dstate", ctypes.c_int32), ("chunk", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


class GdnDims(ctypes.Structure):
    _fields_ = [("nheads", ctypes.c_int32), ("ngroups", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("window", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


class GdnCache(ctypes.Structure):
    _fields_ = [("anchor", ctypes.c_void_p), ("read_copy", ctypes.c_void_p), ("buf_k", ctypes.c_void_p),
                ("buf_v", ctypes.c_void_p), ("buf_g", ctypes.c_void_p), ("buf_beta", ctypes.c_void_p),
                ("buf_u", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("nslots", ctypes.c_int32)]


class ConvDims(ctypes.Structure):
    _fields_ = [("channels", ctypes.c_int32), ("width", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


CONV_SILU = 1


class Params(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p)]


class Cache(ctypes.Structure):
    _fields_ = [("state", ctypes.c_void_p), ("read_copy", ctypes.c_void_p), ("buf_x", ctypes.c_void_p),
                ("buf_dt", ctypes.c_void_p), ("buf_B", ctypes.c_void_p), ("buf_C", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("nslots", ctypes.c_int32), ("read_dtype", ctypes.c_int32),
                ("read_scale", ctypes.c_void_p), ("read_block_scale", ctypes.c_void_p),
                ("anchor_dtype", ctypes.c_int32), ("sr_key", ctypes.c_uint32 * 2), ("sr_nonce", ctypes.c_uint32),
                ("buf_pages", ctypes.c_void_p), ("page_rows", ctypes.c_int32), ("npages", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_U32 = ctypes.c_uint32
_DIMS = ctypes.POINTER(Dims)
_PRM = ctypes.POINTER(Params)
_CACHE = ctypes.POINTER(Cache)

_SIGS = {
    "ers_status_str": ([_I32], ctypes.c_char_p),
    "ers_version": ([], _I32),
    "ers_selftest_bounded_wait": ([ctypes.c_uint64, _P, _P], _I32),
    "ers_ssd_scan_fwd_workspace_size": ([_DIMS, _I32, _I32], _SZ),
    "ers_chunked_prefill_workspace_size": ([_DIMS, _I32, _I32], _SZ),
    "ers_ssd_scan_fwd": ([_DIMS, _PRM, _I32, _I64, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], _I32),
    "ers_ssd_scan_fwd_static": ([_DIMS, _PRM, _I32, _I64, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I32),
    "ers_chunked_prefill": ([_DIMS, _PRM, _CACHE, _I32, _I64, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P],
                            _I32),
    "ers_replay_decode": ([_DIMS, _PRM, _CACHE, _I32, _P, _P, _P, _P, _P, _U32, _P, _P, _P], _I32),
    "ers_refresh": ([_DIMS, _PRM, _CACHE, _I32, _P, _U32, _I32, _P, _P], _I32),
    "ers_spec_verify": ([_DIMS, _PRM, _CACHE, _I32, _P, _I32, _P, _P, _P, _P, _U32, _P, _P, _P], _I32),
    "ers_commit": ([_DIMS, _CACHE, _I32, _P, _P, _I32, _U32, _P, _P], _I32),
    "ers_spec_verify_exact_workspace_size": ([_DIMS, _I32], _SZ),
    "ers_spec_verify_exact": ([_DIMS, _PRM, _CACHE, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], _I32),
    "ers_commit_exact": ([_DIMS, _PRM, _CACHE, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P, _P], _I32),
    "ers_ssu_update": ([_DIMS, _PRM, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P], _I32),
    "ers_conv1d_fwd": ([ctypes.POINTER(ConvDims), _I32, _I64, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _P, _P, _P],
                       _I32),
    "ers_conv1d_update": ([ctypes.POINTER(ConvDims), _I32, _P, _P, _P, _P, _I32, _P, _P, _P, _P], _I32),
    "ers_gdn_verify": ([ctypes.POINTER(GdnDims), ctypes.POINTER(GdnCache), _I32, _P, _I32, _P, _P, _P, _P, _P,
                        _U32, _P, _P, _P], _I32),
    "ers_gdn_commit": ([ctypes.POINTER(GdnDims), ctypes.POINTER(GdnCache), _I32, _P, _P, _I32, _U32, _P, _P], _I32),
    "ers_gdn_refresh": ([ctypes.POINTER(GdnDims), ctypes.POINTER(GdnCache), _I32, _P, _I32, _P, _P], _I32),
}


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name in EXPORTS:
                fn = getattr(L, name)  # AttributeError if the symbol is missing
                fn.argtypes, fn.restype = _SIGS[name]
            _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().ers_status_str(int(code)).decode()


def check(code: int, where: str) -> None:
    if code != ERS_OK:
        raise ErsError(code, where)
