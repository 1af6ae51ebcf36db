"""Python binding of the C ABI in include/mlp_chain.h: argument marshalling only.

Every step of the chain runs in the CUDA library; this module passes device pointers
(``tensor.data_ptr()``) and the CUDA stream handle through ctypes. torch is used only to
obtain those pointers and streams.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import _lib
from ._lib import ChainDesc, ChainInfo, Event, Scoreboard

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT, ERR_DEVICE_STATE, ERR_BAD_TILE = range(8)
DT_BF16, DT_F32 = 1, 2
MODES = {"pipelined": 0, "sequential": 1, "microbatch": 2, "pipelined_kwait": 3, "pipelined_lamport": 4,
         "sequential_pdl": 5}
DEBUG_EVENT_LOG, DEBUG_DROP_DECREMENT, DEBUG_FORCE_RELOAD = 1, 2, 4

EVENT_DTYPE = np.dtype([("stage", np.int32), ("tile", np.int32), ("smid", np.int32), ("cta", np.int32),
                        ("t_start", np.uint64), ("t_end", np.uint64), ("seq_start", np.uint32),
                        ("seq_end", np.uint32), ("t_acc", np.uint64)])


class MlpChainError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = _lib.load().mlp_status_str(int(status)).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


def _check(status: int, what: str):
    if status != OK:
        raise MlpChainError(status, what)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


class Chain:
    """One handle of the library: a fixed chain shape, tile shape and launch mode.

    Shapes follow the header: X[M x dims[0]], W[s][dims[s] x dims[s+1]] (weight_layout "kn") or
    W[s][dims[s+1] x dims[s]] ("nk", nn.Linear's layout), Y[M x dims[-1]].  With ``gated`` the
    first GEMM is SwiGLU and run() takes one more weight: [W_gate, W_up, W_2, ...].

    ``mode`` (every mode gives bit-identical Y for the same tiles):
      "pipelined"          one persistent grid, scoreboard counters and work-queue (CTA-pipelining);
      "pipelined_kwait"    one persistent grid, consumers wait per 64-deep k block of their input;
      "pipelined_lamport"  the queue protocol without fences, consumers validate a sentinel;
      "sequential"         one launch per GEMM;
      "sequential_pdl"     one launch per GEMM, each a programmatic dependent launch of the one before;
      "microbatch"         row chunks of ``microbatch_rows``, GEMMs of different chunks overlapped.
    ``tile_n`` / ``k_split`` per GEMM (0 or None: library choice).  ``cta_pair=2`` runs 256-row
    tiles on CTA pairs (tcgen05 cta_group::2).  ``splitk_exchange`` ("global" or "dsmem") is
    the path split-K siblings add their partial sums through.  ``tile_k=128`` fills the ring with
    two 64-deep k blocks at a time where a GEMM allows it (``info()["fill_k"]``).  ``split_clusters``
    (0 library, 1 one cluster per tile, 2 a cluster per k-slice) places a split tile's k-slices.  Errors raise MlpChainError with
    the library's status.
    """

    def __init__(self, M: int, dims: Sequence[int], *, tile_n: Optional[Sequence[int]] = None,
                 gelu: bool = False, residual: bool = False, mode: str = "pipelined",
                 microbatch_rows: int = 0, device: int = 0, event_log: bool = False,
                 drop_tile: Optional[int] = None, timeout_us: int = 0, grid_ctas: int = 0,
                 raster_group: int = 0, tile_m: int = 0, pipe_stages: int = 0, acc_split: int = 0,
                 weight_layout: str = "kn", k_split: Optional[Sequence[int]] = None, gated: bool = False,
                 force_reload: bool = False, cta_pair: int = 0, splitk_exchange: str = "global",
                 tile_k: int = 0, split_clusters: int = 0):
        lib = _lib.load()
        d = ChainDesc()
        d.M = int(M)
        d.num_gemms = len(dims) - 1
        for i, v in enumerate(dims):
            d.dims[i] = int(v)
        d.in_dtype, d.acc_dtype, d.h_dtype, d.out_dtype = DT_BF16, DT_F32, DT_BF16, DT_BF16
        d.tile_m = int(tile_m)
        for i, v in enumerate(tile_n or []):
            d.tile_n[i] = int(v)
        d.tile_k = int(tile_k)
        d.epilogue = 1 if gelu else 0
        d.residual = int(bool(residual))
        d.mode = MODES[mode]
        d.microbatch_rows = int(microbatch_rows)
        d.device = int(device)
        flags = (DEBUG_EVENT_LOG if event_log else 0) | (DEBUG_FORCE_RELOAD if force_reload else 0)
        if drop_tile is not None:
            flags |= DEBUG_DROP_DECREMENT
            d.drop_tile = int(drop_tile)
        d.debug_flags = flags
        d.timeout_us = int(timeout_us)
        d.grid_ctas = int(grid_ctas)
        d.raster_group = int(raster_group)
        d.pipe_stages = int(pipe_stages)
        d.acc_split = int(acc_split)
        d.weight_layout = {"kn": 0, "nk": 1}[weight_layout]
        for i, v in enumerate(k_split or []):
            d.k_split[i] = int(v)
        d.gated = int(bool(gated))
        d.cta_pair = int(cta_pair)
        d.splitk_exchange = {"global": 1, "dsmem": 2}[splitk_exchange]
        d.split_clusters = int(split_clusters)
        self.M, self.dims, self.mode = int(M), tuple(int(v) for v in dims), mode
        self.n_weights = len(self.dims) - 1 + int(bool(gated))
        self._lib = lib
        h = ctypes.c_void_p()
        _check(lib.mlp_chain_create(ctypes.byref(d), ctypes.byref(h)), "mlp_chain_create")
        self._h = h
        self._wbuf = (ctypes.c_void_p * len(self.dims))()

    # ------------------------------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            self._lib.mlp_chain_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ------------------------------------------------------------------------------------
    def workspace_size(self) -> int:
        n = ctypes.c_size_t()
        _check(self._lib.mlp_chain_workspace_size(self._h, ctypes.byref(n)), "workspace_size")
        return n.value

    def _wptrs(self, Ws):
        if len(Ws) != self.n_weights:
            raise ValueError(f"expected {self.n_weights} weight tensors, got {len(Ws)}")
        for i, w in enumerate(Ws):
            self._wbuf[i] = w.data_ptr() if hasattr(w, "data_ptr") else int(w)
        return self._wbuf

    def run(self, X, Ws, Y, workspace, stream=None):
        """Enqueue the chain; X, Ws, Y, workspace are CUDA tensors (or raw device addresses)."""
        ptr = lambda t: (t.data_ptr() if hasattr(t, "data_ptr") else int(t)) if t is not None else None
        _check(self._lib.mlp_chain_run(self._h, ptr(X), self._wptrs(Ws), ptr(Y), ptr(workspace),
                                       _stream_ptr(stream)), "mlp_chain_run")

    def run_host(self, X_host, Ws, Y_host, X_dev, Y_dev, workspace, stream=None):
        """Enqueue the H2D copy of X_host, the chain, and the transfer into Y_host (page-locked Y_host:
        stored directly by the last GEMM; otherwise through Y_dev and a copy)."""
        ptr = lambda t: t.data_ptr() if hasattr(t, "data_ptr") else int(t)
        _check(self._lib.mlp_chain_run_host(self._h, ptr(X_host), self._wptrs(Ws), ptr(Y_host), ptr(X_dev),
                                            ptr(Y_dev), ptr(workspace) if workspace is not None else None,
                                            _stream_ptr(stream)), "mlp_chain_run_host")

    def check(self, stream=None) -> int:
        """Synchronise and return the device status (0 = OK); re-arms the handle after an error."""
        return int(self._lib.mlp_chain_check(self._h, _stream_ptr(stream)))

    def deps(self, boundary: int = 0):
        off, tgt, init = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        P, C = ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.mlp_chain_get_deps(self._h, boundary, ctypes.byref(off), ctypes.byref(tgt),
                                            ctypes.byref(init), ctypes.byref(P), ctypes.byref(C)), "get_deps")
        offa = np.ctypeslib.as_array(ctypes.cast(off, ctypes.POINTER(ctypes.c_int32)), (P.value + 1,)).copy()
        nnz = int(offa[-1])
        tgta = (np.ctypeslib.as_array(ctypes.cast(tgt, ctypes.POINTER(ctypes.c_int32)), (nnz,)).copy()
                if nnz else np.zeros(0, np.int32))
        inita = np.ctypeslib.as_array(ctypes.cast(init, ctypes.POINTER(ctypes.c_int32)), (C.value,)).copy()
        return offa, tgta, inita

    def scoreboard(self, boundary: int = 0) -> dict:
        """The scoreboard tables the kernel waits on at this stage boundary, read back from the
        device (mlp_chain_get_scoreboard): see _scoreboard_arrays for the keys."""
        return _scoreboard_arrays(lambda sb: self._lib.mlp_chain_get_scoreboard(self._h, boundary, ctypes.byref(sb)),
                                  "get_scoreboard")

    def _full_log(self):
        info = self.info()
        tiles = sum(info["tiles_m"][s] * info["tiles_n"][s] for s in range(info["num_gemms"]))
        cap = tiles + info["grid_ctas"]
        buf = np.zeros(cap, dtype=EVENT_DTYPE)
        n = ctypes.c_size_t()
        _check(self._lib.mlp_chain_get_event_log(self._h, buf.ctypes.data, cap, ctypes.byref(n)), "event_log")
        return buf[: n.value], tiles

    def event_log(self) -> np.ndarray:
        """One record per tile of the last pipelined run (event_log=True)."""
        buf, tiles = self._full_log()
        return buf[:tiles]

    def cta_log(self) -> np.ndarray:
        """One record per CTA of the last pipelined run: t_start = entry, t_acc = set-up done,
        t_end = exit (stage = -1)."""
        buf, tiles = self._full_log()
        return buf[tiles:]

    def info(self) -> dict:
        i = ChainInfo()
        _check(self._lib.mlp_chain_get_info(self._h, ctypes.byref(i)), "get_info")
        S = i.num_gemms
        return {"num_gemms": S, "tile_m": i.tile_m, "tile_k": i.tile_k, "tile_n": list(i.tile_n[:S]),
                "tiles_m": list(i.tiles_m[:S]), "tiles_n": list(i.tiles_n[:S]), "grid_ctas": i.grid_ctas,
                "num_sms": i.num_sms, "pipe_stages": i.pipe_stages, "smem_bytes": i.smem_bytes,
                "tmem_cols": i.tmem_cols, "launches_per_run": i.launches_per_run,
                "cluster_size": i.cluster_size, "k_split": list(i.k_split[:S]), "cta_pair": i.cta_pair,
                "raster_group": i.raster_group, "fill_k": list(i.fill_k[:S]), "split_across": list(i.split_across[:S]),
                "queue_free": list(i.queue_free[:max(S - 1, 0)])}


def deps_build(M: int, n_out: int, n_next: int, bm_p: int, bn_p: int, bm_c: int, bn_c: int):
    """Host-only dependency-array builder (mlp_deps_build): (prod_off, prod_tgt, init_count)."""
    lib = _lib.load()
    P = -(-M // bm_p) * -(-n_out // bn_p)
    C = -(-M // bm_c) * -(-n_next // bn_c)
    init = np.zeros(C, dtype=np.int32)
    nnz = lib.mlp_deps_build(M, n_out, n_next, bm_p, bn_p, bm_c, bn_c, None, None, 0, init.ctypes.data)
    if nnz < 0:
        raise MlpChainError(ERR_INVALID_ARG, "mlp_deps_build")
    off = np.zeros(P + 1, dtype=np.int32)
    tgt = np.zeros(max(nnz, 1), dtype=np.int32)
    r = lib.mlp_deps_build(M, n_out, n_next, bm_p, bn_p, bm_c, bn_c, off.ctypes.data, tgt.ctypes.data,
                           tgt.shape[0], init.ctypes.data)
    if r != nnz:
        raise MlpChainError(ERR_INVALID_ARG, "mlp_deps_build")
    return off, tgt[:nnz], init


def _scoreboard_arrays(call, what: str) -> dict:
    """Two calls of an mlp_scoreboard filler: sizes, then the arrays.  Keys: producers, consumers,
    groups, releases_per_producer, pg_off, pg_tgt, grp_off, grp_mem, grp_target, cons_grp."""
    sb = Scoreboard()
    _check(call(sb), what)
    arr = {"pg_off": np.zeros(sb.producers + 1, np.int32), "pg_tgt": np.zeros(max(sb.edges, 1), np.int32),
           "grp_off": np.zeros(sb.groups + 1, np.int32), "grp_mem": np.zeros(max(sb.consumers, 1), np.int32),
           "grp_target": np.zeros(max(sb.groups, 1), np.int32), "cons_grp": np.zeros(max(sb.consumers, 1), np.int32)}
    for k, a in arr.items():
        setattr(sb, k, a.ctypes.data)
    _check(call(sb), what)
    sizes = {"pg_tgt": sb.edges, "grp_mem": sb.consumers, "grp_target": sb.groups, "cons_grp": sb.consumers}
    out = {k: (a[: sizes[k]] if k in sizes else a) for k, a in arr.items()}
    out.update(producers=sb.producers, consumers=sb.consumers, groups=sb.groups,
               releases_per_producer=sb.releases_per_producer)
    return out


def scoreboard_build(M: int, n_out: int, n_next: int, bm: int, bn_p: int, bn_c: int, raster_group: int = 1,
                     releases_per_producer: int = 4) -> dict:
    """Host-only scoreboard builder (mlp_scoreboard_build), the routine mlp_chain_create uses."""
    lib = _lib.load()
    return _scoreboard_arrays(lambda sb: lib.mlp_scoreboard_build(M, n_out, n_next, bm, bn_p, bn_c, raster_group,
                                                                  releases_per_producer, ctypes.byref(sb)),
                              "mlp_scoreboard_build")


def protocol_model(tiles_m: int, tiles_n: Sequence[int], threads: int = 8, seed: int = 0,
                   drop_tile: int = -1, timeout_ms: int = 2000, return_order: bool = False,
                   raster_group: int = 1, releases_per_tile: int = 4, slices: Optional[Sequence[int]] = None,
                   drop_exchange: int = -1):
    """Run the host-thread protocol model (mlp_protocol_model, or mlp_protocol_model_slices when
    `slices` gives per-stage k-slice counts); returns (status, order), one order entry per item."""
    lib = _lib.load()
    tn = np.ascontiguousarray(tiles_n, dtype=np.int32)
    if slices is None and drop_exchange < 0:
        order = np.full(int(tiles_m * tn.sum()), -1, dtype=np.int32) if return_order else None
        order_ptr = order.ctypes.data if order is not None else None
        st = lib.mlp_protocol_model(len(tn), tiles_m, tn.ctypes.data, raster_group, releases_per_tile, threads, seed,
                                    drop_tile, timeout_ms, order_ptr)
        return int(st), order
    sl = np.ascontiguousarray(slices if slices is not None else [1] * len(tn), dtype=np.int32)
    if sl.shape != tn.shape:
        raise ValueError("slices needs one entry per stage")
    order = np.full(int(tiles_m * (tn * sl).sum()), -1, dtype=np.int32) if return_order else None
    order_ptr = order.ctypes.data if order is not None else None
    st = lib.mlp_protocol_model_slices(len(tn), tiles_m, tn.ctypes.data, sl.ctypes.data, raster_group,
                                       releases_per_tile, threads, seed, drop_tile, drop_exchange, timeout_ms,
                                       order_ptr)
    return int(st), order


NOALLOC_SCRATCH_BYTES = 16 << 20


def run_noalloc(X, W1, W2, Y, sync_check: bool = True, stream=None):
    """mlp_chain_run_noalloc: the two-GEMM chain with no device allocation (all scratch in the
    library's static device array). For callers that may not allocate device memory while they
    run; overlapping calls race. Raises MlpChainError on a non-OK status."""
    lib = _lib.load()
    M, K = X.shape
    N1, N2 = W1.shape[1], W2.shape[1]
    _check(lib.mlp_chain_run_noalloc(M, K, N1, N2, X.data_ptr(), W1.data_ptr(), W2.data_ptr(), Y.data_ptr(),
                                     int(bool(sync_check)), _stream_ptr(stream)), "mlp_chain_run_noalloc")
