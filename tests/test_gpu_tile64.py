"""GPU parity of 64-row tiles (tcgen05 MMAs with M = 64) through the C ABI.

A 64-row accumulator occupies the first 16 lanes of each 32-lane TMEM sub-partition, so every
epilogue warp stores 16 rows.  Bar: within |d| <= 1e-2 (|ref| + 1) of the oracle; bit-exact on
integer-valued inputs; bit-identical across launch modes at the same tiles, including
micro-batch chunks of 64 rows; the scoreboard equals the one rebuilt from the oracle's
enumeration at 64-row tiles; the event log shows every dependency respected.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from test_gpu_chain import DEV, assert_close_to_oracle, bits, run_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mc():
    import mlp_latency_gb300
    mlp_latency_gb300.build()
    mlp_latency_gb300.load()
    return mlp_latency_gb300


def test_tiny_workload_runs_64_by_64_tiles(mc, oracle_mod):
    """The tiny workload's own tiling: 64 x 64 tiles, four producers per consumer."""
    w = si.WORKLOADS["tiny_m64_d256"]
    X, Ws = si.draw(w, seed=0)
    Y, H, info = run_chain(mc, X, Ws, tile_m=64, tile_n=[64, 64])
    assert info["tile_m"] == 64 and info["tiles_m"] == [1, 1] and info["tiles_n"] == [4, 4]
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    with mc.Chain(w.M, w.dims, tile_m=64, tile_n=[64, 64]) as ch:
        off, tgt, init = ch.deps(0)
        assert init.tolist() == [4, 4, 4, 4]


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
@pytest.mark.parametrize("M", [64, 200, 321])
def test_tile_widths_and_ragged_rows_match_oracle(mc, oracle_mod, bn, M):
    X, Ws = si.draw(si.make_workload("t", M, (320, 512, 264)), seed=31)
    Y, H, info = run_chain(mc, X, Ws, tile_m=64, tile_n=[bn, bn], k_split=[1, 1])
    assert info["tiles_m"][0] == -(-M // 64)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)


def test_integer_valued_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(200, (1024, 1024, 512), seed=32)
    Y, H, _ = run_chain(mc, X, Ws, tile_m=64, tile_n=[128, 64])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


@pytest.mark.parametrize("M,dims,tn,ks", [(256, (512, 1024, 256), [128, 64], [1, 1]),
                                          (128, (1024, 2048, 1024), [128, 128], [4, 4]),   # DSMEM split-K
                                          (192, (512, 512, 512), [256, 256], [2, 2])])      # 256 wide
def test_modes_are_bit_identical_at_64_rows(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=33)
    kw = dict(tile_m=64, tile_n=tn, k_split=ks)
    Yp, _, info = run_chain(mc, X, Ws, **kw)
    assert info["tile_m"] == 64
    assert_close_to_oracle(Yp, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))
    for mode in ("sequential", "sequential_pdl", "pipelined_kwait", "pipelined_lamport"):
        Y, _, _ = run_chain(mc, X, Ws, mode=mode, **kw)
        assert torch.equal(Yp.view(torch.int16), Y.view(torch.int16)), mode
    if max(ks) > 1:   # 64-row split tiles up to 256 wide also fit the shared-memory exchange
        Yd, _, _ = run_chain(mc, X, Ws, splitk_exchange="dsmem", **kw)
        assert torch.equal(Yp.view(torch.int16), Yd.view(torch.int16))
    for rows in (64, 128):
        if rows < M:
            Ym, _, info = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=rows, **kw)
            assert info["launches_per_run"] == 2 * -(-M // rows)
            assert torch.equal(Yp.view(torch.int16), Ym.view(torch.int16)), rows


def test_split_8_of_256_wide_tiles(mc, oracle_mod):
    # a 256-wide split tile of 64 rows (64 KB of fp32 partials) reduces through the owners' shared
    # memory, in slices of 32 columns per sibling
    X, Ws = si.draw(si.make_workload("t", 100, (2048, 512, 1024)), seed=34)
    Y, _, info = run_chain(mc, X, Ws, tile_m=64, tile_n=[256, 256], k_split=[8, 4])
    assert info["k_split"] == [8, 4]
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_gated_and_gelu_residual_at_64_rows(mc, oracle_mod):
    M, dims = 130, (256, 512, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims, gated=True), seed=35)
    from test_gpu_swiglu import run_gated
    Y, _ = run_gated(mc, X, Ws, dims, tile_m=64, tile_n=[64, 64])
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gated=True))
    X, Ws = si.draw(si.make_workload("t", M, (256, 256, 256, 256), gelu=True, residual=True), seed=36)
    Y, _, _ = run_chain(mc, X, Ws, tile_m=64, gelu=True, residual=True, tile_n=[64, 128, 64])
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True))


@pytest.mark.parametrize("M,rg", [(576, 0), (1088, 3)])
def test_scoreboard_and_event_log_at_64_rows(mc, oracle_mod, M, rg):
    import expected_scoreboard as es
    dims, tn = (256, 512, 384), [64, 128]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=37)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_m=64, tile_n=tn, event_log=True, raster_group=rg) as ch:
        info = ch.info()
        tm = info["tiles_m"][0]
        g = info["raster_group"]
        assert (g == rg) if rg else (g == 8 if tm >= 16 else g == 4 if tm >= 8 else g in (1, tm))
        es.assert_equal(ch.scoreboard(0), es.expected(oracle_mod, M, dims[1], dims[2], 64, tn[0], tn[1], g, 4))
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        for _ in range(2):
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
            ev = ch.event_log()
            off, tgt, _ = ch.deps(0)
            p_end = {int(e["tile"]): int(e["seq_end"]) for e in ev if e["stage"] == 0}
            c_start = {int(e["tile"]): int(e["seq_start"]) for e in ev if e["stage"] == 1}
            assert len(p_end) == tm * info["tiles_n"][0] and len(c_start) == tm * info["tiles_n"][1]
            for p in range(len(off) - 1):
                for c in tgt[off[p]:off[p + 1]]:
                    assert p_end[p] < c_start[int(c)]
    assert_close_to_oracle(Y.cpu(), oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_decode_workload_at_64_rows_sampled(mc, oracle_mod):
    """The decode workload (M = 128) as two 64-row panels, in the pipelined and micro-batched
    (64-row chunks) modes, on sampled rows of the oracle."""
    w = si.WORKLOADS["decode_m128_d4096"]
    X, Ws = si.draw(w, seed=0)
    Yp, _, _ = run_chain(mc, X, Ws, tile_m=64)
    Ym, _, info = run_chain(mc, X, Ws, tile_m=64, mode="microbatch", microbatch_rows=64)
    assert info["launches_per_run"] == 4
    assert torch.equal(Yp.view(torch.int16), Ym.view(torch.int16))
    rows = si.sample_rows(w.M, 16, seed=5)
    Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws], rows=rows)
    assert_close_to_oracle(Yp[rows], Yo)
