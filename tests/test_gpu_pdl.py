"""GPU parity of MLP_MODE_SEQUENTIAL_PDL through the C ABI: one launch per GEMM, each later one a
programmatic dependent launch of the one before (its TMA warp waits for the previous grid with
griddepcontrol.wait before loading that grid's output).

Only when each launch's loads may start changes, never the tiles or the k order: Y and every
intermediate must be bit-identical to MLP_MODE_SEQUENTIAL, also when the runs are captured in a
CUDA graph (where the dependency becomes a programmatic graph edge), and within
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


@pytest.mark.parametrize("M,dims,tn,ks", [
    (64, (256, 256, 256), [64, 64], None),
    (300, (512, 384, 512), [64, 128], [1, 2]),        # ragged rows, split-K in the second GEMM
    (128, (1024, 1024, 1024), [128, 128], [4, 4]),    # clusters of 4 in both launches
    (257, (1000, 328, 96), None, None),               # ragged K and N, library tiles
])
def test_pdl_bit_identical_to_sequential(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=81)
    Yp, Hp, info = run_chain(mc, X, Ws, mode="sequential_pdl", tile_n=tn, k_split=ks)
    assert info["launches_per_run"] == len(dims) - 1
    Ys, Hs, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=ks)
    assert same(Yp, Ys) and same(Hp, Hs)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(Hp, Ho)
    assert_close_to_oracle(Yp, Yo)


def test_pdl_four_gemm_gelu_residual_chain(mc, oracle_mod):
    # three dependent launches: GEMM s + 2 waits on s + 1, which waited on s
    w = si.make_workload("t", 300, (512,) * 5, gelu=True, residual=True)
    X, Ws = si.draw(w, seed=82)
    kw = dict(gelu=True, residual=True, tile_n=[64, 128, 64, 128])
    Yp, _, _ = run_chain(mc, X, Ws, mode="sequential_pdl", **kw)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", **kw)
    assert same(Yp, Ys)
    assert_close_to_oracle(Yp, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True))


def test_pdl_repeated_runs_and_graph_replay_at_decode_size(mc):
    w = si.WORKLOADS["decode_m128_d4096"]
    X, Ws = si.draw(w, seed=0)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential")
    outs, _, _ = run_chain(mc, X, Ws, mode="sequential_pdl", reps=3)
    for o in outs:
        assert same(o, Ys)
    Xd, Wd = X.to(DEV), [t.to(DEV) for t in Ws]
    with mc.Chain(w.M, w.dims, mode="sequential_pdl") as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(w.M, w.dims[-1], dtype=torch.bfloat16, device=DEV)
        stream = torch.cuda.Stream()
        ch.run(Xd, Wd, Y, ws, stream=stream)           # encode the maps before capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            ch.run(Xd, Wd, Y, ws, stream=stream)
        for _ in range(3):
            Y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert ch.check() == 0
            assert same(Y.cpu(), Ys)
