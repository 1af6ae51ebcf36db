"""GPU parity of CTA-pair tiles (tcgen05 cta_group::2, `cta_pair=2`) through the C ABI.

A pair computes a 256-row tile: each CTA loads its 128 rows of the activations and half of the
weight tile's columns, the leader issues every MMA and each CTA's TMEM holds its 128 rows.  A
split-K tile takes one pair per k-slice; each CTA adds the slices of its own rows with the
same-half CTAs of the other pairs, through global memory.  Bar:
within |d| <= 1e-2 (|ref| + 1) of the oracle; bit-exact on integer-valued inputs; bit-identical
to single-CTA tiles of the same width (the same 16-deep dot products in the same order) and
across launch modes; the scoreboard equals the one rebuilt from the oracle's enumeration at
256-row tiles, and the event log shows every dependency respected.
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


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,dims,tn", [
    (256, (512, 512, 256), [256, 256]),       # one pair tile per column
    (300, (320, 264, 520), [256, 128]),       # the second pair tile: 44 rows, the peer's half all past M
    (640, (1024, 768, 384), [128, 256]),      # 3 pair-row panels, 128-wide tiles (64 columns per CTA)
    (129, (64, 128, 64), [128, 128]),         # one row past the leader's half; narrow outputs
])
def test_pairs_match_oracle_and_single_cta_tiles(mc, oracle_mod, M, dims, tn):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=41)
    Yp, Hp, info = run_chain(mc, X, Ws, tile_n=tn, cta_pair=2, k_split=[1, 1])
    assert info["cta_pair"] == 2 and info["tile_m"] == 256 and info["cluster_size"] == 2
    assert info["tiles_m"][0] == -(-M // 256)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(Hp, Ho)
    assert_close_to_oracle(Yp, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, tile_n=tn, k_split=[1, 1])
    assert same(Yp, Ys)


def test_pairs_integer_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(300, (1024, 1024, 512), seed=42)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[256, 256], cta_pair=2)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


@pytest.mark.parametrize("M,dims,tn", [(1024, (512, 1024, 512), [256, 256]), (600, (256, 384, 256), [128, 256])])
def test_pair_modes_are_bit_identical(mc, M, dims, tn):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=43)
    kw = dict(tile_n=tn, cta_pair=2)
    Yp, _, _ = run_chain(mc, X, Ws, **kw)
    for mode in ("sequential", "sequential_pdl"):
        Y, _, _ = run_chain(mc, X, Ws, mode=mode, **kw)
        assert same(Yp, Y), mode
    for rows in (256, 512):
        if rows < M:
            Y, _, info = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=rows, **kw)
            assert info["launches_per_run"] == 2 * -(-M // rows)
            assert same(Yp, Y), rows


def test_pairs_gelu_residual_four_gemm_chain(mc, oracle_mod):
    M, dims = 700, (256, 512, 384, 256, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims, gelu=True, residual=True), seed=44)
    Y, _, _ = run_chain(mc, X, Ws, gelu=True, residual=True, cta_pair=2)
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True))
    Ys, _, _ = run_chain(mc, X, Ws, gelu=True, residual=True, mode="sequential", cta_pair=2)
    assert same(Y, Ys)


@pytest.mark.parametrize("M,rg", [(1280, 0), (4352, 0), (2304, 3)])
def test_pair_scoreboard_and_event_log(mc, oracle_mod, M, rg):
    import expected_scoreboard as es
    dims, tn = (256, 512, 256), [256, 128]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=45)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, event_log=True, raster_group=rg, cta_pair=2, k_split=[1, 1]) as ch:
        info = ch.info()
        tm = info["tiles_m"][0]
        g = info["raster_group"]
        assert (g == rg) if rg else (g == 8 if tm >= 16 else g == 4 if tm >= 8 else g in (1, tm))
        es.assert_equal(ch.scoreboard(0), es.expected(oracle_mod, M, dims[1], dims[2], 256, tn[0], tn[1], g, 8))
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


def test_pairs_many_runs_and_nk_weights(mc, oracle_mod):
    M, dims = 1100, (512, 768, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=46)
    outs, _, _ = run_chain(mc, X, Ws, reps=20, cta_pair=2)
    for o in outs[1:]:
        assert same(o, outs[0])
    Wt = [w.t().contiguous() for w in Ws]   # nn.Linear layout: N x K
    Yt, _, _ = run_chain(mc, X, Wt, weight_layout="nk", cta_pair=2)
    assert same(Yt, outs[0])
    assert_close_to_oracle(outs[0], oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_prefill_workload_on_pairs_sampled(mc, oracle_mod):
    w = si.WORKLOADS["prefill_m2048_d8192"]
    X, Ws = si.draw(w, seed=0)
    Y, _, info = run_chain(mc, X, Ws, cta_pair=2)
    assert info["tile_n"] == [256, 256] and info["cta_pair"] == 2
    rows = si.sample_rows(w.M, 24, seed=6)
    assert_close_to_oracle(Y[rows], oracle_mod.chain(bits(X), [bits(t) for t in Ws], rows=rows))


@pytest.mark.parametrize("M,dims,tn,ks", [
    (256, (2048, 1024, 512), [256, 256], [4, 4]),    # clusters of 8: four pairs per tile
    (300, (1024, 512, 264), [128, 256], [2, 1]),     # ragged rows and columns, mixed splits
    (700, (3072, 640, 384), [256, 128], [2, 4]),     # three pair-row panels, ragged N, the last k-slice 1 block
])
def test_pairs_with_split_k_match_oracle_and_single_cta_tiles(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=47)
    Yp, Hp, info = run_chain(mc, X, Ws, tile_n=tn, k_split=ks, cta_pair=2)
    assert info["cta_pair"] == 2 and info["k_split"] == ks and info["cluster_size"] == 2 * max(ks)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(Hp, Ho)
    assert_close_to_oracle(Yp, Yo)
    # the same k-slices added in the same order: bit-identical to one CTA per tile
    Ys, Hs, info1 = run_chain(mc, X, Ws, tile_n=tn, k_split=ks, cta_pair=1)
    assert info1["cta_pair"] == 1
    assert same(Hp, Hs) and same(Yp, Ys)
    for mode in ("sequential", "sequential_pdl"):
        Y, _, _ = run_chain(mc, X, Ws, mode=mode, tile_n=tn, k_split=ks, cta_pair=2)
        assert same(Yp, Y), mode
    Ym, _, _ = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=256, tile_n=tn, k_split=ks, cta_pair=2)
    assert same(Yp, Ym)
    outs, _, _ = run_chain(mc, X, Ws, reps=6, tile_n=tn, k_split=ks, cta_pair=2)
    for o in outs:
        assert same(o, Yp)


def test_pair_split_k_integer_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(256, (2048, 512, 1024), seed=48)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[256, 128], k_split=[4, 2], cta_pair=2)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_pair_split_k_scoreboard_and_event_log(mc, oracle_mod):
    """Each CTA of a split pair tile releases its rows once per epilogue warp: 2 x S x 4 releases
    per producer tile, against the groups rebuilt from the oracle's enumeration."""
    import expected_scoreboard as es
    M, dims, tn, ks = 1024, (1024, 512, 1024), [256, 128], [2, 4]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=49)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, k_split=ks, event_log=True, cta_pair=2) as ch:
        info = ch.info()
        tm = info["tiles_m"][0]
        g = info["raster_group"]
        es.assert_equal(ch.scoreboard(0), es.expected(oracle_mod, M, dims[1], dims[2], 256, tn[0], tn[1], g, 2 * ks[0] * 4))
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


def test_pairs_refuse_more_than_four_k_slices(mc):
    """A split pair tile takes 2 x k_split CTAs of one cluster, at most 8."""
    with pytest.raises(mc.MlpChainError) as e:
        mc.Chain(256, (4096, 512, 512), tile_n=[256, 256], k_split=[8, 1], cta_pair=2)
    assert e.value.status == mc.ERR_UNSUPPORTED


def test_llama_workload_library_choice_sampled(mc, oracle_mod):
    """The Llama MLP (one 256-row panel) with the library's tiling, on sampled rows."""
    w = si.WORKLOADS["llama_m256_4096_14336"]
    X, Ws = si.draw(w, seed=0)
    Y, _, info = run_chain(mc, X, Ws)
    rows = si.sample_rows(w.M, 16, seed=7)
    assert_close_to_oracle(Y[rows], oracle_mod.chain(bits(X), [bits(t) for t in Ws], rows=rows))
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=info["tile_n"], k_split=info["k_split"],
                         cta_pair=info["cta_pair"])
    assert same(Y, Ys)


@pytest.mark.parametrize("ks", [[1, 1], [1, 2]])
def test_pair_dropped_release_times_out_then_recovers(mc, ks):
    """Two pair panels, a pair for every consumer item (a queue-free boundary: the consumer pairs
    send their first weight copies, then wait on their group's counter).  Producer tile 1 withholds
    its releases, so the consumers of its panel run out of time: both CTAs of each such pair send
    the activation copies of their armed fills anyway, the run ends in TIMEOUT, and the next run
    (the fault fires once) gives the sequential launches' bits."""
    M, dims = 512, (1024, 1024, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=23)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    kw = dict(tile_n=[128, 128], k_split=ks, cta_pair=2, raster_group=1)
    with mc.Chain(M, dims, drop_tile=1, timeout_us=20000, **kw) as ch:
        assert ch.info()["queue_free"] == [1] and ch.info()["cta_pair"] == 2
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == mc.ERR_TIMEOUT
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == 0
        Y2 = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", **kw)
    assert same(Y2, Ys)
