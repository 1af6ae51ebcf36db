"""GPU parity of split-K slices on separate clusters (`split_clusters=2`, CTA pairs).

Every k-slice of a split pair tile is a cluster item of its own (a pair); the slices exchange their
partial sums through buffers of their own in global memory, count their releases on one counter
per tile and half, and add the parts in slice order, as the in-cluster exchange does.  Bar: within
|d| <= 1e-2 (|ref| + 1) of the oracle; bit-exact on integer-valued inputs; bit-identical to the
same tiles and slices in one cluster and to the sequential launches; the device scoreboard equal to
the tables rebuilt from the oracle's enumeration; every dependency respected in the event log;
forty runs of one handle give the same bits.
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


@pytest.mark.parametrize("M,dims,tn,ks", [
    (256, (2048, 2048, 1024), [256, 256], [1, 4]),    # the down-projection split four ways
    (256, (1024, 1536, 768), [128, 256], [2, 2]),     # both GEMMs split (the first: static items)
    (200, (1000, 1024, 520), [256, 128], [1, 2]),     # ragged rows, K and N; uneven k-slices
    (96, (512, 2048, 512), [256, 256], [2, 4]),       # a peer half wholly past M
])
def test_separate_cluster_slices_match_oracle_and_one_cluster(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=91)
    kw = dict(tile_n=tn, k_split=ks, cta_pair=2)
    Y, H, info = run_chain(mc, X, Ws, split_clusters=2, **kw)
    assert info["cta_pair"] == 2 and info["cluster_size"] == 2
    assert info["split_across"] == [int(k > 1) for k in ks]
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Y1, H1, info1 = run_chain(mc, X, Ws, split_clusters=1, **kw)
    assert info1["split_across"] == [0, 0] and info1["cluster_size"] == 2 * max(ks)
    assert same(Y, Y1) and same(H, H1)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", **kw)
    assert same(Y, Ys)


@pytest.mark.parametrize("M,dims,tn,ks", [
    (256, (1024, 1536, 768), [128, 256], [2, 2]),   # the producer's slices on separate clusters
    (256, (2048, 2048, 1024), [256, 256], [1, 4]),  # only the consumer's
])
def test_scoreboard_matches_oracle_enumeration(mc, oracle_mod, M, dims, tn, ks):
    """Each slice's pair releases its rows once per epilogue warp, wherever the slices run:
    2 x S x 4 releases per producer tile, against the groups rebuilt from the oracle's
    enumeration of overlapping tiles."""
    import expected_scoreboard as es
    with mc.Chain(M, dims, tile_n=tn, k_split=ks, cta_pair=2, split_clusters=2) as ch:
        info = ch.info()
        assert info["split_across"] == [int(k > 1) for k in ks]
        es.assert_equal(ch.scoreboard(0), es.expected(oracle_mod, M, dims[1], dims[2], 256, tn[0], tn[1],
                                                      info["raster_group"], 2 * ks[0] * 4))


def test_integer_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(256, (2048, 1024, 1024), seed=92)
    Y, H, _ = run_chain(mc, X, Ws, split_clusters=2, tile_n=[256, 256], k_split=[2, 4], cta_pair=2)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_many_runs_and_event_log(mc):
    """The per-tile counters accumulate over runs against the run's epoch: forty runs give the
    same bits; in an event-logged run every consumer starts after all of its producers."""
    M, dims = 256, (1024, 2048, 1024)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=93)
    kw = dict(split_clusters=2, tile_n=[256, 256], k_split=[2, 4], cta_pair=2)
    outs, _, _ = run_chain(mc, X, Ws, reps=40, **kw)
    for o in outs[1:]:
        assert same(o, outs[0])
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, event_log=True, **kw) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == 0
        ev = ch.event_log()
        off, tgt, _ = ch.deps(0)
    p_end = {int(e["tile"]): int(e["seq_end"]) for e in ev if e["stage"] == 0}
    c_start = {int(e["tile"]): int(e["seq_start"]) for e in ev if e["stage"] == 1}
    assert len(p_end) == 8 and len(c_start) == 4
    for p in range(len(off) - 1):
        for c in tgt[off[p]:off[p + 1]]:
            assert p_end[p] < c_start[int(c)]
    assert same(Y.cpu(), outs[0])


def test_dropped_release_times_out_then_recovers(mc):
    M, dims = 256, (1024, 1024, 1024)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=94)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    kw = dict(split_clusters=2, tile_n=[256, 256], k_split=[2, 4], cta_pair=2)
    with mc.Chain(M, dims, drop_tile=1, timeout_us=20000, **kw) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == mc.ERR_TIMEOUT
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == 0
        Y2 = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=[256, 256], k_split=[2, 4], cta_pair=2)
    assert same(Y2, Ys)


def test_requests_the_layout_cannot_run_are_refused(mc):
    with pytest.raises(mc.MlpChainError):   # two 256-row panels
        mc.Chain(512, (1024, 1024, 1024), split_clusters=2, cta_pair=2, tile_n=[256, 256], k_split=[1, 4])
    with pytest.raises(mc.MlpChainError):   # 64 tiles x 4 slices: more items than clusters of two
        mc.Chain(256, (4096, 4096, 16384), split_clusters=2, cta_pair=2, tile_n=[256, 256], k_split=[1, 4])
