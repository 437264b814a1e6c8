"""ctypes binding of libzl_attn.so (the C ABI in include/zl_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  If the library has not been built this module raises on import of
the functions that need it; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libzl_attn.so")

ZL_OK = 0
ZL_EINVAL = -1
ZL_EUNSUPPORTED = -2
ZL_EALIGN = -3
ZL_EWORKSPACE = -4
ZL_ECUDA = -5
ZL_ETIMEOUT = -6
ZL_ENODEVICE = -7

ZL_BF16 = 0
ZL_FP32 = 1

# Every symbol include/zl_attn.h declares.
EXPORTS = (
    "zl_status_string", "zl_version", "zl_varlen_attn_fwd_workspace_size", "zl_varlen_attn_fwd",
    "zl_lse_merge", "zl_varlen_attn_bwd_workspace_size", "zl_varlen_attn_bwd", "zl_sync_check",
    "zl_launch_count", "zl_profile_begin", "zl_profile_end", "zl_varlen_attn_bwd_static",
    "zl_varlen_attn_fwd_ex", "zl_lse_merge_ex", "zl_varlen_attn_fwd_schedule", "zl_varlen_attn_bwd_schedule",
    "zl_selftest_wait_timeout",
)

ZL_FWD_FUSED_MERGE = 1
ZL_FWD_BF16_PARTIALS = 2


class WorkItem(ctypes.Structure):
    """zl_work_item_t"""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("launch", "seq", "tile", "head", "q_start", "q_len", "k_start", "k_len")]


class BwdWorkItem(ctypes.Structure):
    """zl_bwd_work_item_t"""
    _fields_ = [(n, ctypes.c_int32) for n in ("launch", "seq", "head", "k_start", "k_len", "q_len")]


class Tile(ctypes.Structure):
    """zl_tile_t"""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("seq", "q_start", "q_len", "k_start", "k_len", "q_chunk", "kv_chunk", "n_kv_chunks",
                 "h_start", "h_len", "h_chunk")]


class ProfileEntry(ctypes.Structure):
    """zl_profile_entry_t"""
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class ZlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib = None


def load() -> ctypes.CDLL:
    """Loads the in-tree library (building it is build()'s job)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run `python -m mixed_length_dit_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    c_i32, c_i64, c_f32, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    vp = ctypes.c_void_p
    i32p = ctypes.POINTER(ctypes.c_int32)
    tilep = ctypes.POINTER(Tile)
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.zl_status_string.restype = ctypes.c_char_p
    lib.zl_status_string.argtypes = [c_i32]
    lib.zl_version.restype = c_i32
    lib.zl_version.argtypes = []
    lib.zl_launch_count.restype = c_i64
    lib.zl_launch_count.argtypes = []
    lib.zl_sync_check.restype = c_i32
    lib.zl_sync_check.argtypes = [vp]
    lib.zl_selftest_wait_timeout.restype = c_i32
    lib.zl_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.zl_varlen_attn_fwd_workspace_size.restype = c_i32
    lib.zl_varlen_attn_fwd_workspace_size.argtypes = [i32p, i32p, c_i32, c_i32, c_i32, tilep, c_i32, szp]
    lib.zl_varlen_attn_fwd.restype = c_i32
    lib.zl_varlen_attn_fwd.argtypes = [vp, vp, vp, i32p, i32p, c_i32, c_i32, c_i32, c_i32, c_f32,
                                       tilep, c_i32, vp, vp, vp, c_sz, vp]
    lib.zl_varlen_attn_fwd_ex.restype = c_i32
    lib.zl_varlen_attn_fwd_ex.argtypes = [vp, vp, vp, i32p, i32p, c_i32, c_i32, c_i32, c_i32, c_f32,
                                          tilep, c_i32, vp, vp, vp, c_sz, vp, ctypes.c_uint32]
    lib.zl_lse_merge.restype = c_i32
    lib.zl_lse_merge.argtypes = [vp, vp, c_i32, c_i64, c_i32, c_i32, c_i64, vp, c_i32, vp, c_i64, vp]
    lib.zl_varlen_attn_fwd_schedule.restype = c_i32
    lib.zl_varlen_attn_fwd_schedule.argtypes = [i32p, i32p, c_i32, c_i32, c_i32, c_i32, tilep, c_i32,
                                                ctypes.POINTER(WorkItem), c_i64, ctypes.POINTER(c_i64)]
    lib.zl_varlen_attn_bwd_schedule.restype = c_i32
    lib.zl_varlen_attn_bwd_schedule.argtypes = [i32p, i32p, c_i32, c_i32, c_i32, tilep, c_i32,
                                                ctypes.POINTER(BwdWorkItem), c_i64, ctypes.POINTER(c_i64)]
    lib.zl_lse_merge_ex.restype = c_i32
    lib.zl_lse_merge_ex.argtypes = [vp, c_i32, vp, c_i32, c_i64, c_i32, c_i32, c_i64, vp, c_i32, vp, c_i64, vp]
    lib.zl_varlen_attn_bwd_workspace_size.restype = c_i32
    lib.zl_varlen_attn_bwd_workspace_size.argtypes = [i32p, i32p, c_i32, c_i32, c_i32, szp]
    lib.zl_varlen_attn_bwd.restype = c_i32
    lib.zl_varlen_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i32p, i32p, c_i32, c_i32, c_i32, c_i32,
                                       c_f32, tilep, c_i32, vp, vp, vp, vp, c_sz, vp]
    lib.zl_profile_begin.restype = c_i32
    lib.zl_profile_begin.argtypes = []
    lib.zl_profile_end.restype = c_i32
    lib.zl_profile_end.argtypes = [ctypes.POINTER(ProfileEntry), c_i32, ctypes.POINTER(c_i32)]
    lib.zl_varlen_attn_bwd_static.restype = c_i32
    lib.zl_varlen_attn_bwd_static.argtypes = [vp, vp, vp, vp, vp, vp, i32p, i32p, c_i32, c_i32, c_i32,
                                              c_f32, vp, vp, vp, vp]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().zl_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != ZL_OK:
        raise ZlError(status, where)


def int32_array(values):
    """Host int32 array for cu_seqlens (list, tuple, numpy or CPU tensor)."""
    vals = [int(x) for x in (values.tolist() if hasattr(values, "tolist") else values)]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals), len(vals)


def tile_array(tiles):
    """Host zl_tile_t array from tuples (seq, q_start, q_len, k_start, k_len,
    q_chunk, kv_chunk, n_kv_chunks[, h_start, h_len, h_chunk]); a tuple of
    eight leaves the head range zero, i.e. all heads."""
    if not tiles:
        return None, 0
    arr = (Tile * len(tiles))()
    names = [f[0] for f in Tile._fields_]
    for i, t in enumerate(tiles):
        if len(t) not in (8, 11):
            raise ValueError("a tile has 8 or 11 fields")
        for name, val in zip(names, t):
            setattr(arr[i], name, int(val))
    return arr, len(tiles)
