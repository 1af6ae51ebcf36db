"""CPU-only checks of the C ABI library: it builds, loads, exports every declared symbol, and
its host logic (dependency-array builder, protocol model, argument validation) is right.
No call here touches a GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import mlp_latency_gb300 as mc
from mlp_latency_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mc.build()
    return mc.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mlp_chain.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mlp_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no binding"


def test_struct_layouts_match_the_c_compiler(tmp_path):
    """Offsets of every ctypes field equal the C compiler's offsetof for the header's structs."""
    structs = {"mlp_chain_desc": _lib.ChainDesc, "mlp_event": _lib.Event, "mlp_chain_info": _lib.ChainInfo}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mlp_chain.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                          check=True).stdout.split("\n") if l)
    for cname, cls in structs.items():
        assert int(out[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(out[f"{cname}.{f}"]) == getattr(cls, f).offset, f"{cname}.{f}"


def test_status_strings(lib):
    for s in range(8):
        assert lib.mlp_status_str(s)


SHAPES = [
    (64, 256, 256, 64, 64, 64, 64),
    (64, 256, 256, 128, 64, 128, 64),
    (128, 4096, 4096, 128, 32, 128, 32),
    (300, 192, 160, 128, 64, 128, 32),
    (300, 200, 100, 64, 48, 128, 64),
    (257, 96, 64, 128, 32, 64, 64),
    (1, 64, 64, 128, 64, 128, 64),
    (513, 128, 384, 128, 128, 128, 256),
    (2048, 1024, 512, 128, 256, 128, 128),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_deps_builder_matches_oracle_enumeration(lib, oracle_mod, shape):
    off, tgt, init = mc.deps_build(*shape)
    o_off, o_tgt, o_init = oracle_mod.deps(*shape)
    assert np.array_equal(off, o_off)
    assert np.array_equal(tgt, o_tgt)
    assert np.array_equal(init, o_init)


def test_tiny_config_has_four_producers_per_consumer(lib):
    # 64 rows, 64x64 tiles: one row panel, 4 producer and 4 consumer tiles
    off, tgt, init = mc.deps_build(64, 256, 256, 128, 64, 128, 64)
    assert init.tolist() == [4, 4, 4, 4]
    assert off.tolist() == [0, 4, 8, 12, 16]


@pytest.mark.parametrize("tiles_m,tiles_n,threads,seed,rg,rel", [
    (1, [4, 4], 4, 0, 1, 4), (4, [8, 3], 8, 1, 1, 16), (3, [5, 7, 2, 4], 6, 2, 1, 4), (6, [2, 9], 16, 3, 1, 8),
    (2, [1, 1], 3, 4, 1, 4), (9, [4, 5], 8, 5, 4, 8), (17, [3, 2, 3], 12, 6, 8, 4), (7, [2, 6], 6, 7, 3, 32),
    # no more consumer tiles than threads: queue-free boundaries of several groups
    (4, [3, 2], 8, 8, 1, 4), (3, [4, 3, 2], 9, 9, 1, 8), (4, [2, 4], 16, 10, 2, 4),
])
def test_protocol_model_orders_every_tile(lib, tiles_m, tiles_n, threads, seed, rg, rel):
    """Merged raster groups, several releases per tile, counters accumulating over three runs."""
    st, order = mc.protocol_model(tiles_m, tiles_n, threads=threads, seed=seed, return_order=True,
                                  raster_group=rg, releases_per_tile=rel)
    assert st == mc.OK
    total = tiles_m * sum(tiles_n)
    assert sorted(order.tolist()) == sorted((s << 24) | t for s in range(len(tiles_n))
                                            for t in range(tiles_m * tiles_n[s]))


@pytest.mark.parametrize("rg", [1, 4])
def test_protocol_model_dropped_decrement_times_out(lib, rg):
    st, _ = mc.protocol_model(8 if rg > 1 else 2, [4, 4], threads=4, seed=5, drop_tile=1, timeout_ms=200,
                              raster_group=rg)
    assert st == mc.ERR_TIMEOUT


def test_protocol_model_dropped_decrement_times_out_without_queue(lib):
    # 8 consumer tiles on 8 threads in 4 groups: the consumers skip the queue and wait on their
    # group's counter, which the dropped releases keep short
    st, _ = mc.protocol_model(4, [2, 2], threads=8, seed=6, drop_tile=1, timeout_ms=200)
    assert st == mc.ERR_TIMEOUT


@pytest.mark.parametrize("tiles_m,tiles_n,slices,threads,seed,rg,rel", [
    (2, [4, 4], [2, 1], 16, 11, 1, 8),         # a sliced first stage (static tickets)
    (1, [8, 4], [1, 4], 16, 12, 1, 8),         # a sliced consumer stage after a one-group boundary
    (2, [4, 2, 4], [2, 4, 1], 16, 13, 2, 8),   # both, with merged raster groups
    (4, [3, 2], [1, 2], 16, 14, 1, 4),         # a sliced consumer stage at a queue-free boundary of 4 groups
    (1, [4, 4], [4, 4], 16, 15, 1, 16),        # every stage sliced, 4 releases per slice
    (2, [3, 3], [1, 1], 6, 16, 1, 4),          # no slices through the same entry point
])
def test_protocol_model_slices_on_separate_items(lib, tiles_m, tiles_n, slices, threads, seed, rg, rel):
    """k-slices as items of their own (the device's slices on separate clusters): every slice of
    every tile runs once per run, the exchange counters land on each run's target, and each tile
    appears once per slice in the completion order."""
    st, order = mc.protocol_model(tiles_m, tiles_n, threads=threads, seed=seed, return_order=True,
                                  raster_group=rg, releases_per_tile=rel, slices=slices)
    assert st == mc.OK
    assert sorted(order.tolist()) == sorted((s << 24) | t for s in range(len(tiles_n))
                                            for t in range(tiles_m * tiles_n[s]) for _ in range(slices[s]))


def test_protocol_model_withheld_exchange_times_out(lib):
    # first-stage tile 3's last slice writes its partials but never adds to the tile's exchange
    # counter: its siblings (and it) wait until the deadline
    st, _ = mc.protocol_model(2, [4, 4], threads=16, seed=17, slices=[2, 1], releases_per_tile=8,
                              drop_exchange=3, timeout_ms=200)
    assert st == mc.ERR_TIMEOUT


def test_protocol_model_sliced_tile_withheld_releases_time_out(lib):
    st, _ = mc.protocol_model(2, [4, 4], threads=16, seed=18, slices=[2, 1], releases_per_tile=8,
                              drop_tile=3, timeout_ms=200)
    assert st == mc.ERR_TIMEOUT


@pytest.mark.parametrize("tiles_n,slices,threads,rel,drop_exchange", [
    ([4, 4], [2, 1], 15, 8, -1),   # 16 sliced items on 15 threads: more than one wave
    ([4, 4], [3, 1], 16, 8, -1),   # 3 slices do not divide 8 releases
    ([4, 4], [1, 2], 16, 8, 0),    # a withheld exchange on an unsliced first stage
    ([4, 4], [2, 1], 16, 8, 8),    # ... or on a tile that does not exist
    ([4, 4], [0, 1], 16, 8, -1),
])
def test_protocol_model_slices_rejects_bad_arguments(lib, tiles_n, slices, threads, rel, drop_exchange):
    st, _ = mc.protocol_model(2, tiles_n, threads=threads, slices=slices, releases_per_tile=rel,
                              drop_exchange=drop_exchange)
    assert st == mc.ERR_INVALID_ARG


def _desc(**kw):
    d = _lib.ChainDesc()
    d.M, d.num_gemms = 128, 2
    for i, v in enumerate((256, 256, 256)):
        d.dims[i] = v
    d.in_dtype, d.acc_dtype, d.h_dtype, d.out_dtype = 1, 2, 1, 1
    for k, v in kw.items():
        if k in ("dims", "tile_n", "k_split"):
            for i, x in enumerate(v):
                getattr(d, k)[i] = x
        else:
            setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,expect", [
    ({"num_gemms": 0}, mc.ERR_INVALID_ARG),
    ({"num_gemms": 5}, mc.ERR_INVALID_ARG),
    ({"M": 0}, mc.ERR_INVALID_ARG),
    ({"dims": (256, 100, 256)}, mc.ERR_INVALID_ARG),
    ({"in_dtype": 2}, mc.ERR_UNSUPPORTED),
    ({"tile_m": 96}, mc.ERR_UNSUPPORTED),
    ({"residual": 1, "dims": (256, 256, 512)}, mc.ERR_INVALID_ARG),
    ({"mode": 2, "microbatch_rows": 100}, mc.ERR_INVALID_ARG),
    ({"mode": 6}, mc.ERR_INVALID_ARG),                             # modes 0 .. 5
    ({"mode": 7}, mc.ERR_INVALID_ARG),
    # a gated (SwiGLU) first GEMM keeps gate and up side by side in TMEM: unsplit, <= 128 wide
    ({"gated": 1, "acc_split": 2}, mc.ERR_UNSUPPORTED),
    ({"gated": 1, "k_split": (2, 0)}, mc.ERR_UNSUPPORTED),
    ({"gated": 1, "tile_n": (256, 0)}, mc.ERR_UNSUPPORTED),
    # CTA pairs: no split accumulators, K-granular or Lamport modes; 128 or 256 wide (gated: 64 or 128)
    ({"cta_pair": 3}, mc.ERR_INVALID_ARG),
    ({"splitk_exchange": 3}, mc.ERR_INVALID_ARG),
    ({"splitk_exchange": -1}, mc.ERR_INVALID_ARG),
    ({"cta_pair": 2, "gated": 1, "tile_n": (32, 0)}, mc.ERR_UNSUPPORTED),   # a gated pair tile: 64 or 128 wide
    ({"cta_pair": 2, "splitk_exchange": 2}, mc.ERR_UNSUPPORTED),    # pairs add split-K parts via L2
    ({"cta_pair": 2, "mode": 3}, mc.ERR_UNSUPPORTED),
    ({"cta_pair": 2, "mode": 4}, mc.ERR_UNSUPPORTED),
    ({"cta_pair": 2, "tile_n": (64, 0)}, mc.ERR_UNSUPPORTED),
    ({"cta_pair": 2, "tile_m": 64}, mc.ERR_UNSUPPORTED),
    ({"cta_pair": 2, "mode": 2, "microbatch_rows": 128}, mc.ERR_INVALID_ARG),   # chunks of 256 rows
    # ring fills 64 or 128 deep; two-block fills need one CTA per tile, one accumulator, no
    # per-block consumer work (K-granular waits, Lamport scans)
    ({"tile_k": 96}, mc.ERR_UNSUPPORTED),
    ({"tile_k": 256}, mc.ERR_UNSUPPORTED),
    ({"tile_k": 128, "cta_pair": 2}, mc.ERR_UNSUPPORTED),
    ({"tile_k": 128, "mode": 3}, mc.ERR_UNSUPPORTED),
    ({"tile_k": 128, "mode": 4}, mc.ERR_UNSUPPORTED),
    ({"tile_k": 128, "acc_split": 2}, mc.ERR_UNSUPPORTED),
    # k-slices on separate clusters: the queue protocol on CTA pairs over one 256-row panel
    ({"split_clusters": 3}, mc.ERR_INVALID_ARG),
    ({"split_clusters": -1}, mc.ERR_INVALID_ARG),
    ({"split_clusters": 2, "mode": 1}, mc.ERR_UNSUPPORTED),
    ({"split_clusters": 2, "mode": 3}, mc.ERR_UNSUPPORTED),
    ({"split_clusters": 2, "cta_pair": 1}, mc.ERR_UNSUPPORTED),
    ({"split_clusters": 2, "acc_split": 2}, mc.ERR_UNSUPPORTED),
    ({"split_clusters": 2, "M": 257}, mc.ERR_UNSUPPORTED),
])
def test_create_rejects_bad_descriptors_before_touching_cuda(lib, kw, expect):
    h = ctypes.c_void_p()
    assert lib.mlp_chain_create(ctypes.byref(_desc(**kw)), ctypes.byref(h)) == expect
    assert not h.value


def test_null_arguments(lib):
    assert lib.mlp_chain_create(None, None) == mc.ERR_INVALID_ARG
    assert lib.mlp_chain_run(None, None, None, None, None, None) == mc.ERR_INVALID_ARG
    assert lib.mlp_chain_check(None, None) == mc.ERR_INVALID_ARG
    assert lib.mlp_chain_destroy(None) == mc.ERR_INVALID_ARG


# (M, n_out, n_next, bm, bn_p, bn_c): one row panel, several, ragged M and N, unequal widths
SB_SHAPES = [
    (64, 256, 256, 128, 64, 64),
    (128, 4096, 4096, 128, 128, 128),
    (300, 192, 160, 128, 64, 32),
    (1000, 512, 384, 128, 128, 64),
    (2048, 1024, 512, 128, 256, 128),
    (2100, 640, 256, 128, 256, 256),
    (1, 64, 64, 128, 64, 64),
]


@pytest.mark.parametrize("shape", SB_SHAPES)
@pytest.mark.parametrize("rg", [1, 3, 4, 8])
@pytest.mark.parametrize("releases", [4, 16])
def test_scoreboard_matches_oracle_enumeration(lib, oracle_mod, shape, rg, releases):
    """The grouped counters and their targets (what the consumer prologue waits on) equal the ones
    rebuilt from the oracle's brute-force tile-overlap enumeration, element by element."""
    import expected_scoreboard as es
    got = mc.scoreboard_build(*shape, raster_group=rg, releases_per_producer=releases)
    es.assert_equal(got, es.expected(oracle_mod, *shape, rg, releases))


def test_scoreboard_decode_is_one_group_waiting_for_every_release(lib):
    # M = 128: one row panel, every consumer depends on all 32 producers, each releasing S x 4 times
    sb = mc.scoreboard_build(128, 4096, 4096, 128, 128, 128, raster_group=1, releases_per_producer=16)
    assert sb["groups"] == 1 and sb["grp_target"].tolist() == [32 * 16]
    assert sb["grp_mem"].tolist() == list(range(32))


def test_scoreboard_build_rejects_bad_arguments(lib):
    sb = _lib.Scoreboard()
    assert lib.mlp_scoreboard_build(128, 256, 256, 128, 64, 64, 1, 4, None) == mc.ERR_INVALID_ARG
    assert lib.mlp_scoreboard_build(0, 256, 256, 128, 64, 64, 1, 4, ctypes.byref(sb)) == mc.ERR_INVALID_ARG
    assert lib.mlp_scoreboard_build(128, 256, 256, 128, 0, 64, 1, 4, ctypes.byref(sb)) == mc.ERR_INVALID_ARG
    assert lib.mlp_scoreboard_build(128, 256, 256, 128, 64, 64, 1, 0, ctypes.byref(sb)) == mc.ERR_INVALID_ARG
    assert lib.mlp_chain_get_scoreboard(None, 0, ctypes.byref(sb)) == mc.ERR_INVALID_ARG
