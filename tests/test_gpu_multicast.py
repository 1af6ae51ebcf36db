"""GPU parity of A-tile multicast clusters (mlp_chain_desc.a_multicast) through the C ABI.

Each CTA of a cluster loads 1/n of the activation tile and multicasts it to the cluster; every
MMA commit frees the slot in all n CTAs.  Only where the tiles are read from changes, so Y must
be bit-identical to the same tiles without multicast and to the sequential launches, and within
|d| <= 1e-2 (|ref| + 1) of the oracle.
"""
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


@pytest.mark.parametrize("M,dims,tn,n", [
    (128, (1024, 1024, 512), [32, 32], 4),
    (100, (512, 1024, 1024), [64, 32], 8),     # ragged rows: the pieces past M are zero-filled
    (128, (2048, 512, 256), [64, 64], 2),
])
@pytest.mark.parametrize("mode", ["pipelined", "pipelined_kwait", "sequential"])
def test_multicast_matches_plain_tiles_and_oracle(mc, oracle_mod, M, dims, tn, n, mode):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=61)
    Y, H, info = run_chain(mc, X, Ws, mode=mode, tile_n=tn, k_split=[1, 1], a_multicast=n)
    assert info["cluster_size"] == n
    Yp, _, _ = run_chain(mc, X, Ws, mode=mode, tile_n=tn, k_split=[1, 1])
    assert same(Y, Yp)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)


def test_multicast_repeats_and_full_size_decode(mc, oracle_mod):
    # the same tiles without split-K sum in the same order: bit-identical to sequential launches
    w = si.WORKLOADS["decode_m128_d4096"]
    X, Ws = si.draw(w, seed=0)
    kw = dict(tile_n=[32, 32], k_split=[1, 1])
    outs, _, _ = run_chain(mc, X, Ws, reps=3, a_multicast=4, **kw)
    for o in outs[1:]:
        assert same(o, outs[0])
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", **kw)
    assert same(outs[0], Ys)
    rows = si.sample_rows(w.M, 16, seed=6)
    Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws], rows=rows)
    assert_close_to_oracle(outs[0][torch.as_tensor(rows)], Yo)


@pytest.mark.parametrize("M,dims,kw", [
    (256, (512, 512, 512), dict(tile_n=[64, 64])),                             # two row panels
    (128, (512, 512, 512), dict(tile_n=[64, 64], k_split=[2, 1])),             # a split stage
    (128, (512, 320, 512), dict(tile_n=[64, 64])),                             # 5 column tiles
    (128, (512, 512, 512), dict(tile_n=[64, 64], mode="pipelined_lamport")),   # re-loads per CTA
])
def test_multicast_rejects_what_it_cannot_share(mc, M, dims, kw):
    with pytest.raises(mc.MlpChainError):
        mc.Chain(M, dims, a_multicast=4, **kw)
