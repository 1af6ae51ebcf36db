"""GPU parity of the K-granular pipelined mode (MLP_MODE_PIPELINED_KWAIT) through the C ABI.

The mode changes only when a consumer's k blocks may be loaded (each waits for the producer
tiles that wrote those columns, instead of for its whole producer set through the work-queue),
never the arithmetic: Y must be bit-identical to the sequential launches and within
|d| <= 1e-2 (|ref| + 1) of the oracle; integer-valued inputs are bit-exact.
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
    (64, (256, 256, 256), [64, 64], None),             # one producer tile per k block
    (300, (256, 384, 512), [32, 128], None),           # producer tiles narrower than a k block
    (512, (512, 1024, 256), [256, 64], None),          # four k blocks per producer tile
    (128, (1024, 1024, 1024), [128, 128], [4, 4]),     # split-K producers and consumers
    (257, (1000, 328, 96), None, None),                # ragged edges, library choice
])
def test_kwait_matches_oracle_and_sequential(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=31)
    Y, H, _ = run_chain(mc, X, Ws, mode="pipelined_kwait", tile_n=tn, k_split=ks)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=ks)
    assert same(Y, Ys)
    Yp, _, _ = run_chain(mc, X, Ws, mode="pipelined", tile_n=tn, k_split=ks)
    assert same(Y, Yp)


def test_kwait_integer_inputs_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(256, (1024, 512, 1024), seed=32)
    Y, H, _ = run_chain(mc, X, Ws, mode="pipelined_kwait", tile_n=[64, 128], k_split=[2, 4])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_kwait_four_gemm_gelu_residual_chain(mc, oracle_mod):
    # the middle stages consume and produce: each waits per k block and releases its rows
    w = si.make_workload("t", 300, (512,) * 5, gelu=True, residual=True)
    X, Ws = si.draw(w, seed=33)
    kw = dict(gelu=True, residual=True, tile_n=[64, 128, 64, 128])
    Y, _, _ = run_chain(mc, X, Ws, mode="pipelined_kwait", **kw)
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True))
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", **kw)
    assert same(Y, Ys)


def test_kwait_repeated_runs_accumulate_ready_counts(mc):
    # ready counters are never cleared between runs: run e waits for (e + 1) x quota releases
    X, Ws = si.draw(si.make_workload("t", 384, (512, 512, 256)), seed=34)
    outs, _, _ = run_chain(mc, X, Ws, mode="pipelined_kwait", reps=6, tile_n=[64, 64], k_split=[2, 1])
    for o in outs[1:]:
        assert same(o, outs[0])


@pytest.mark.parametrize("grid,ks,tn", [(2, [1, 1], [64, 64]), (4, [2, 2], [64, 64])])
def test_kwait_small_grid_still_completes(mc, oracle_mod, grid, ks, tn):
    # far fewer CTAs than tiles: consumers hold tickets only after every producer's ticket
    X, Ws = si.draw(si.make_workload("t", 512, (256, 512, 256)), seed=35)
    Y, _, info = run_chain(mc, X, Ws, mode="pipelined_kwait", grid_ctas=grid, k_split=ks, tile_n=tn)
    assert info["grid_ctas"] == grid
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_kwait_withheld_release_times_out_then_recovers(mc):
    M, dims = 256, (512, 512, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=36)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, mode="pipelined_kwait", tile_n=[64, 64], k_split=[2, 1], drop_tile=3,
                  timeout_us=20000) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)                    # tile 3 never counts itself ready
        assert ch.check() == mc.ERR_TIMEOUT      # ... so the consumers reading it time out
        for _ in range(2):                       # check() cleared the counters and the epoch
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
        Y2 = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=[64, 64], k_split=[2, 1])
    assert same(Y2, Ys)


@pytest.mark.parametrize("name", ["decode_m128_d4096", "llama_m256_4096_14336"])
def test_kwait_full_size_is_bit_identical_to_queue_protocol(mc, name):
    w = si.WORKLOADS[name]
    X, Ws = si.draw(w, seed=0)
    Yk, _, info = run_chain(mc, X, Ws, mode="pipelined_kwait")
    # the same tiles and k-slices (the queue protocol may otherwise run them on CTA pairs, which
    # compute the same bits: see the pair tests)
    Yp, _, _ = run_chain(mc, X, Ws, mode="pipelined", tile_n=info["tile_n"], k_split=info["k_split"])
    assert same(Yk, Yp)
