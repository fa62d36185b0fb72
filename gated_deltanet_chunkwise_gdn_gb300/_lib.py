"""ctypes loader for libgdn_gb300.so (the C ABI of include/gdn.h).

There is no fallback: if the library cannot be loaded (or built), every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS_NAMES = {
    0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_BAD_INDEX",
    4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_TIMEOUT", 6: "GDN_ERR_CUDA", 7: "GDN_ERR_BAD_SEQLENS",
}
GDN_BF16, GDN_FP16 = 0, 1


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load the shared library (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libgdn_gb300.so not found at {path}; run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        i32, i64, f32, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        L.gdn_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32, i32]
        L.gdn_workspace_size.restype = sz
        L.gdn_extend_chunkwise.argtypes = [
            vp, vp, vp, ctypes.c_int,      # q k v dtype
            vp, vp, vp, vp,                # a b A_log dt_bias
            vp, i64, vp, vp, i32,          # state_pool pool_size cache_indices cu_seqlens batch
            vp, i64, i32, i32, i32, i32,   # out total_tokens H HV K V
            i32, f32, vp, sz, vp]          # chunk_size scale workspace bytes stream
        L.gdn_extend_chunkwise.restype = ctypes.c_int
        L.gdn_extend_chunkwise_noalloc.argtypes = [
            vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, i64, vp, vp, i32,
            vp, i64, i32, i32, i32, i32, i32, f32, vp, vp]
        L.gdn_extend_chunkwise_noalloc.restype = ctypes.c_int
        L.gdn_backward_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32, i32]
        L.gdn_backward_workspace_size.restype = sz
        L.gdn_chunkwise_backward.argtypes = [
            vp, vp, vp, ctypes.c_int,      # q k v dtype
            vp, vp, vp, vp,                # a b A_log dt_bias
            vp, i64, vp, vp, i32,          # state_pool pool_size cache_indices cu_seqlens batch
            vp, vp,                        # d_out d_state
            vp, vp, vp, vp, vp, vp, vp, vp,  # dq dk dv da db dA_log ddt_bias d_state_pool
            i64, i32, i32, i32, i32,       # total_tokens H HV K V
            i32, f32, vp, sz, vp]          # chunk_size scale workspace bytes stream
        L.gdn_chunkwise_backward.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [
            vp, vp, vp, ctypes.c_int,      # q k v dtype
            vp, vp, vp, vp,                # a b A_log dt_bias
            vp, i64, vp, i32, vp,          # state_pool pool_size cache_indices batch out
            i32, i32, i32, i32, f32,       # H HV K V scale
            vp, vp]                        # device_status stream
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_get_device_status.argtypes = [vp, vp]
        L.gdn_get_device_status.restype = ctypes.c_int
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_profile_start.argtypes = [i32]
        L.gdn_profile_start.restype = ctypes.c_int
        L.gdn_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64), i32]
        L.gdn_profile_stop.restype = i32
        L.gdn_kernel_name.argtypes = [i32]
        L.gdn_kernel_name.restype = ctypes.c_char_p
        L.gdn_launch_count.argtypes = []
        L.gdn_launch_count.restype = i64
        L.gdn_version.argtypes = []
        L.gdn_version.restype = i32
        L.gdn_workspace_layout.argtypes = [i64, i32, i32, i32, i32, i32, i32, ctypes.POINTER(WorkspaceLayout)]
        L.gdn_workspace_layout.restype = ctypes.c_int
        L.gdn_test_set_stall.argtypes = [i32, i64]
        L.gdn_test_set_stall.restype = ctypes.c_int
        _lib = L
        return L


class WorkspaceLayout(ctypes.Structure):
    """gdn_workspace_layout_t of include/gdn.h (byte offsets of the per-chunk intermediates)."""
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "chunk_tab", "g", "beta", "rq", "rk", "ks", "w", "u", "p",
                                                "seg_state", "seg_map", "total")] + [
        ("max_chunks", ctypes.c_int64), ("block", ctypes.c_int32), ("affine_factors", ctypes.c_int32),
        ("nseg", ctypes.c_int32)]


def workspace_layout(total_tokens: int, batch: int, H: int, HV: int, K: int, V: int, chunk_size: int):
    lay = WorkspaceLayout()
    check(load().gdn_workspace_layout(total_tokens, batch, H, HV, K, V, chunk_size, ctypes.byref(lay)),
          "gdn_workspace_layout")
    return lay


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def check(status: int, what: str):
    if status != 0:
        raise GdnError(status, f"{what}: {status_string(status)}")
