"""ctypes binding of libmuon's C ABI (include/muon.h): marshalling only.

Every function here forwards to the library with the same name; there is no
computation and no fallback.  If libmuon.so has not been built the first use
raises, so a missing extension can never turn into a silent CPU path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmuon.so")

MUON_OK = 0
MUON_ERR_INVALID_ARG = -1
MUON_ERR_UNSUPPORTED = -2
MUON_ERR_NO_WORKSPACE = -3
MUON_ERR_CUDA = -4
MUON_ERR_TIMEOUT = -5
MUON_ERR_STATE = -6
MUON_F32 = 0
MUON_BF16 = 1
MUON_FULL = 0
MUON_BLOCKWISE = 1
MUON_DISTRIBUTED = 2
MUON_HOST_ONLY = -1
MUON_N_STAGES = 8
STAGE_NAMES = ("momentum", "norm", "normalise", "syrk1", "syrk2", "gemm",
               "update", "chain")

# Every entry point include/muon.h declares.
EXPORTS = ("muon_create", "muon_set_stream", "muon_register_params",
           "muon_workspace_size", "muon_set_workspace", "muon_step",
           "muon_sync", "muon_destroy", "muon_last_error",
           "muon_set_profiling", "muon_stage_times", "muon_last_launch_count",
           "muon_debug_set_exports", "muon_get_plan_info",
           "muon_step_noalloc", "muon_debug_wait_timeout", "muon_step_host",
           "muon_debug_check_chain_schedule", "muon_debug_set_chain_test",
           "muon_dist_configure", "muon_dist_momentum", "muon_dist_gram",
           "muon_dist_update")


class MuonParam(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("g", ctypes.c_void_p),
                ("m", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld_w", ctypes.c_int64),
                ("ld_g", ctypes.c_int64), ("ld_m", ctypes.c_int64),
                ("w_dtype", ctypes.c_int32), ("g_dtype", ctypes.c_int32)]


class MuonPlanInfo(ctypes.Structure):
    _fields_ = [("units", ctypes.c_int64), ("groups", ctypes.c_int64),
                ("syrk_tiles", ctypes.c_int64), ("gemm_tiles", ctypes.c_int64),
                ("ew_tiles", ctypes.c_int64),
                ("useful_flops", ctypes.c_int64),
                ("executed_flops", ctypes.c_int64),
                ("chained_groups", ctypes.c_int64)]


class MuonError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libmuon error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmuon.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m newton_schulz_06_gb300.build` (or "
            "__graft_entry__.build()); there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    H = ctypes.c_void_p
    vp = ctypes.c_void_p
    i32 = ctypes.c_int
    f32 = ctypes.c_float
    sz = ctypes.c_size_t
    sig = {
        "muon_create": [ctypes.POINTER(H), i32, vp],
        "muon_set_stream": [H, vp],
        "muon_register_params": [H, i32, ctypes.POINTER(MuonParam)],
        "muon_workspace_size": [H, i32, i32, ctypes.POINTER(sz),
                                ctypes.POINTER(sz)],
        "muon_set_workspace": [H, vp, sz],
        "muon_step": [H, f32, f32, i32, i32, f32, f32, f32, i32, i32],
        "muon_sync": [H],
        "muon_destroy": [H],
        "muon_last_error": [H],
        "muon_set_profiling": [H, i32],
        "muon_stage_times": [H, ctypes.POINTER(f32), ctypes.POINTER(i32),
                             i32],
        "muon_last_launch_count": [H],
        "muon_debug_set_exports": [H, i32, ctypes.POINTER(vp),
                                   ctypes.POINTER(vp)],
        "muon_get_plan_info": [H, i32, i32, ctypes.POINTER(MuonPlanInfo)],
        "muon_step_noalloc": [ctypes.POINTER(MuonParam), f32, f32, i32, i32,
                              f32, f32, f32, vp, ctypes.c_char_p, sz],
        "muon_debug_wait_timeout": [H, vp, i32],
        "muon_debug_check_chain_schedule": [H, i32, i32],
        "muon_debug_set_chain_test": [H, i32],
        "muon_step_host": [H, i32, ctypes.POINTER(vp), ctypes.POINTER(vp), f32,
                           f32, i32, i32, f32, f32, f32, i32, i32],
        "muon_dist_configure": [H, i32, f32],
        "muon_dist_momentum": [H, f32, i32, vp],
        "muon_dist_gram": [H, vp, ctypes.c_int64, i32, i32],
        "muon_dist_update": [H, vp, ctypes.c_int64, i32, i32, vp, f32, f32, f32,
                             f32],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "muon_last_error" else i32
    _lib = L
    return L


def check(rc: int, handle=None) -> int:
    if rc < 0:
        msg = lib().muon_last_error(handle).decode(errors="replace")
        raise MuonError(rc, msg)
    return rc
