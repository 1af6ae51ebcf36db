"""CPU oracle for the CTA-pipelined GEMM chain -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline`` / reference leg may
import this package. The product path (``mlp_latency_gb300``) never imports, loads or calls it,
and this package imports nothing from the product path; the two share only ``seeded_inputs``.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc). This module builds it on demand
and marshals numpy arrays of bf16 bit patterns (``uint16``) through ctypes.

Citations for every function are in ``oracle.c``; in short, after "CTA-Pipelining: A
Latency-Oriented Spatial Scaling Method for Multi-GPU Systems":
  * ``chain``  -- the two-layer GEMM running example (section III) generalised to S layers
    (section IV multi-layer GEMM), bf16 in/out with fp32 accumulation (Fig. 2 set-up);
  * ``deps``   -- the dependency array of section III-A, by brute-force tile-overlap enumeration;
  * ``gelu``   -- GeLU in tanh form, used by the GeLU chain workload (not on the pages).
Every function here has at least one independent pin in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread"]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_liboracle.so (gcc). Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.oracle_chain.restype = ctypes.c_int
            lib.oracle_chain.argtypes = [i64, i32, vp, vp, vp, i32, i32, i32, vp, i64, vp, vp, i32]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_deps.restype = i64
            lib.oracle_deps.argtypes = [i64, i64, i64, i32, i32, i32, i32, vp, vp, i64, vp]
            lib.oracle_gelu_tanh.restype = ctypes.c_double
            lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = None
            lib.oracle_round_bf16.argtypes = [vp, vp, i64]
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    if hasattr(a, "view") and not isinstance(a, np.ndarray):  # torch bf16 tensor
        import torch  # local: only for the conversion
        a = a.contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def chain(X, Ws: Sequence, gelu: bool = False, residual: bool = False,
          rows: Optional[np.ndarray] = None, threads: Optional[int] = None,
          return_h: bool = False, gated: bool = False):
    """Y (and optionally the first intermediate H) of the chain, for all rows or ``rows``.

    X: M x d0 bf16 bits; Ws[s]: d_s x d_{s+1} bf16 bits. With ``gated`` the first stage takes
    two matrices, Ws[0] (gate) and Ws[1] (up), both d0 x d1, and H = SiLU(X Wg) * (X Wu).
    Returns uint16 arrays (len(rows) or M) x d_S, and (..) x d_1 for H.
    """
    lib = _load()
    X = _u16(X)
    Ws = [_u16(w) for w in Ws]
    M = X.shape[0]
    if gated and (len(Ws) < 3 or Ws[0].shape != Ws[1].shape):
        raise ValueError("a gated chain needs gate and up matrices of one shape, then the rest")
    stage_ws = Ws[1:] if gated else Ws
    dims = [X.shape[1]] + [w.shape[1] for w in stage_ws]
    for s, w in enumerate(stage_ws):
        if w.shape[0] != dims[s]:
            raise ValueError(f"W{s + 1} has {w.shape[0]} rows, expected {dims[s]}")
    dims_a = np.array(dims, dtype=np.int64)
    wptrs = (ctypes.c_void_p * len(Ws))(*[w.ctypes.data for w in Ws])
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.shape[0]
    else:
        n = M
    Y = np.empty((n, dims[-1]), dtype=np.uint16)
    H = np.empty((n, dims[1]), dtype=np.uint16) if return_h else None
    rc = lib.oracle_chain(M, len(stage_ws), dims_a.ctypes.data, X.ctypes.data, wptrs, int(gelu),
                          int(residual), int(gated), rows.ctypes.data if rows is not None else None, n,
                          Y.ctypes.data, H.ctypes.data if H is not None else None,
                          threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_chain failed ({rc})")
    return (Y, H) if return_h else Y


def deps(M: int, n_out: int, n_next: int, bm_p: int, bn_p: int, bm_c: int, bn_c: int):
    """(prod_off[P+1], prod_tgt[nnz], init_count[C]) by brute-force tile-overlap enumeration."""
    lib = _load()
    P = -(-M // bm_p) * -(-n_out // bn_p)
    C = -(-M // bm_c) * -(-n_next // bn_c)
    init = np.zeros(C, dtype=np.int32)
    nnz = lib.oracle_deps(M, n_out, n_next, bm_p, bn_p, bm_c, bn_c, None, None, 0, init.ctypes.data)
    if nnz < 0:
        raise RuntimeError(f"oracle_deps failed ({nnz})")
    off = np.zeros(P + 1, dtype=np.int32)
    tgt = np.zeros(max(nnz, 1), dtype=np.int32)
    rc = lib.oracle_deps(M, n_out, n_next, bm_p, bn_p, bm_c, bn_c, off.ctypes.data, tgt.ctypes.data,
                         tgt.shape[0], init.ctypes.data)
    if rc != nnz:
        raise RuntimeError(f"oracle_deps failed ({rc})")
    return off, tgt[:nnz], init


def gelu(x: float) -> float:
    return _load().oracle_gelu_tanh(float(x))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact: shift into the upper half)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def silu(x: float) -> float:
    """The oracle's SiLU, x / (1 + e^-x) in double."""
    return float(_load().oracle_silu(float(x)))
