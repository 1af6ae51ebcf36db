"""Build and load libmlp_chain.so (the CUDA library behind include/mlp_chain.h).

The library is compiled in-tree with nvcc for sm_103a only. Loading it never falls back to
anything else: if the shared object is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libmlp_chain.so")
SOURCES = [os.path.join(CSRC, "mlp_chain.cu"), os.path.join(CSRC, "host_protocol.cpp")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("chain_kernel.cuh", "ptx.cuh", "protocol.h", "dep_groups.h")] + [
    os.path.join(INCLUDE, "mlp_chain.h")]

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-pthread", "-shared", "--threads", "0",
]

_lock = threading.Lock()
_lib = None


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library with nvcc (cross-compiles without a GPU). Returns its path."""
    if force or _stale():
        nvcc = os.environ.get("NVCC", "nvcc")
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc, *NVCC_FLAGS, "-I", INCLUDE, "-o", tmp, *SOURCES]
        if verbose:
            print(" ".join(cmd))
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
vp, szt = ctypes.c_void_p, ctypes.c_size_t
MAX_GEMMS = 4


class ChainDesc(ctypes.Structure):
    _fields_ = [
        ("M", i64), ("num_gemms", i32), ("dims", i64 * (MAX_GEMMS + 1)),
        ("in_dtype", ctypes.c_int), ("acc_dtype", ctypes.c_int), ("h_dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int), ("tile_m", i32), ("tile_n", i32 * MAX_GEMMS), ("tile_k", i32),
        ("epilogue", ctypes.c_int), ("residual", i32), ("mode", ctypes.c_int),
        ("microbatch_rows", i32), ("device", i32), ("debug_flags", u32), ("drop_tile", i32),
        ("timeout_us", u32), ("grid_ctas", i32), ("raster_group", i32), ("pipe_stages", i32),
        ("weight_layout", i32), ("k_split", i32 * MAX_GEMMS), ("acc_split", i32), ("gated", i32), ("cta_pair", i32),
        ("splitk_exchange", i32), ("split_clusters", i32),
    ]


class Event(ctypes.Structure):
    _fields_ = [("stage", i32), ("tile", i32), ("smid", i32), ("cta", i32), ("t_start", u64),
                ("t_end", u64), ("seq_start", u32), ("seq_end", u32), ("t_acc", u64)]


class ChainInfo(ctypes.Structure):
    _fields_ = [
        ("num_gemms", i32), ("tile_m", i32), ("tile_k", i32), ("tile_n", i32 * MAX_GEMMS),
        ("tiles_m", i32 * MAX_GEMMS), ("tiles_n", i32 * MAX_GEMMS), ("grid_ctas", i32),
        ("num_sms", i32), ("pipe_stages", i32), ("smem_bytes", i32), ("tmem_cols", i32),
        ("launches_per_run", i32), ("cluster_size", i32), ("k_split", i32 * MAX_GEMMS), ("cta_pair", i32),
        ("raster_group", i32), ("fill_k", i32 * MAX_GEMMS),
        ("split_across", i32 * MAX_GEMMS), ("queue_free", i32 * MAX_GEMMS),
    ]


class Scoreboard(ctypes.Structure):
    _fields_ = [("producers", i32), ("consumers", i32), ("groups", i32), ("edges", i32),
                ("releases_per_producer", i32), ("pg_off", vp), ("pg_tgt", vp), ("grp_off", vp),
                ("grp_mem", vp), ("grp_target", vp), ("cons_grp", vp)]


# every symbol include/mlp_chain.h declares: name -> (restype, argtypes)
SIGNATURES = {
    "mlp_chain_create": (ctypes.c_int, [ctypes.POINTER(ChainDesc), ctypes.POINTER(vp)]),
    "mlp_chain_workspace_size": (ctypes.c_int, [vp, ctypes.POINTER(szt)]),
    "mlp_chain_run": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
    "mlp_chain_run_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp]),
    "mlp_chain_check": (ctypes.c_int, [vp, vp]),
    "mlp_chain_get_deps": (ctypes.c_int, [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                          ctypes.POINTER(vp), ctypes.POINTER(i32), ctypes.POINTER(i32)]),
    "mlp_scoreboard_build": (ctypes.c_int, [i64, i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(Scoreboard)]),
    "mlp_chain_get_scoreboard": (ctypes.c_int, [vp, i32, ctypes.POINTER(Scoreboard)]),
    "mlp_chain_get_event_log": (ctypes.c_int, [vp, vp, szt, ctypes.POINTER(szt)]),
    "mlp_chain_get_info": (ctypes.c_int, [vp, ctypes.POINTER(ChainInfo)]),
    "mlp_chain_destroy": (ctypes.c_int, [vp]),
    "mlp_deps_build": (i64, [i64, i64, i64, i32, i32, i32, i32, vp, vp, i64, vp]),
    "mlp_protocol_model": (ctypes.c_int, [i32, i32, vp, i32, i32, i32, u64, i32, u32, vp]),
    "mlp_protocol_model_slices": (ctypes.c_int, [i32, i32, vp, vp, i32, i32, i32, u64, i32, i32, u32, vp]),
    "mlp_chain_run_noalloc": (ctypes.c_int, [i64, i64, i64, i64, vp, vp, vp, vp, i32, vp]),
    "mlp_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}


def load():
    """The loaded library. Raises if it has not been built (there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library {LIB_PATH} is missing: call "
                                   "mlp_latency_gb300.build() (needs nvcc) first")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
