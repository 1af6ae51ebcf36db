"""GPU parity of ring fills two k blocks deep (tile_k = 128).

Each fill carries the A and B tiles of two consecutive 64-deep k blocks, one copy per operand
through views whose outermost coordinate is the k block, and the MMA thread issues both blocks'
MMAs from one barrier phase.  The MMAs run in the same k order into the same accumulator as with
one-block fills, so the results are bit-identical to tile_k = 64 at the same tiles and splits.
Bar: within |d| <= 1e-2 (|ref| + 1) of the oracle; bit-identical to one-block fills and across
launch modes; bit-exact on integer-valued inputs.
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
    (128, (1024, 1024, 768), [128, 128], [4, 2]),    # decode-like: one row panel, split-K slices
    (200, (512, 768, 1024), [64, 128], [1, 2]),      # ragged rows
    (384, (768, 512, 256), [256, 32], [1, 1]),       # the widest tile; 32 columns (64-byte boxes)
    (256, (2048, 1536, 512), [96, 128], [1, 4]),     # a width of 1.5 boxes: one-block fills there
])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_deep_fills_match_oracle_and_one_block_fills(mc, oracle_mod, M, dims, tn, ks, layout):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=81)
    Wl = [w.t().contiguous() for w in Ws] if layout == "nk" else Ws
    Y, H, info = run_chain(mc, X, Wl, tile_k=128, tile_n=tn, k_split=ks, cta_pair=1, weight_layout=layout)
    assert info["tile_n"] == tn and info["k_split"] == ks
    whole_boxes = [layout == "nk" or t % 64 == 0 or t == 32 for t in tn]
    assert info["fill_k"] == [128 if w else 64 for w in whole_boxes]
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Y1, H1, info1 = run_chain(mc, X, Wl, tile_k=64, tile_n=tn, k_split=ks, cta_pair=1, weight_layout=layout)
    assert info1["fill_k"] == [64, 64]
    assert same(Y, Y1) and same(H, H1)
    for mode in ("sequential", "sequential_pdl"):
        Ym, _, _ = run_chain(mc, X, Wl, mode=mode, tile_k=128, tile_n=tn, k_split=ks, cta_pair=1,
                             weight_layout=layout)
        assert same(Y, Ym), mode


def test_ring_slots_hold_two_blocks(mc):
    with mc.Chain(128, (1024, 1024, 1024), tile_k=128, tile_n=[128, 128], k_split=[4, 4], cta_pair=1) as ch:
        deep = ch.info()
    with mc.Chain(128, (1024, 1024, 1024), tile_k=64, tile_n=[128, 128], k_split=[4, 4], cta_pair=1) as ch:
        flat = ch.info()
    assert deep["fill_k"] == [128, 128] and deep["tile_k"] == 128
    assert flat["fill_k"] == [64, 64] and flat["tile_k"] == 64
    # a slot of 2 x (16 KB + 16 KB) against 16 KB + 16 KB: about half the slots
    assert deep["pipe_stages"] == flat["pipe_stages"] // 2


@pytest.mark.parametrize("M,dims,ks,want", [
    (128, (576, 512, 512), [1, 1], [64, 128]),       # K = 576 is not a multiple of 128
    (128, (768, 512, 512), [4, 1], [64, 128]),       # 12 blocks in slices of 3
    (128, (512, 1024, 512), [4, 2], [128, 128]),     # slices of 2 blocks: one fill each
])
def test_gemms_that_cannot_fill_deep_fall_back(mc, oracle_mod, M, dims, ks, want):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=82)
    Y, H, info = run_chain(mc, X, Ws, tile_k=128, tile_n=[128, 128], k_split=ks, cta_pair=1)
    assert info["fill_k"] == want
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))
    Y1, _, _ = run_chain(mc, X, Ws, tile_k=64, tile_n=[128, 128], k_split=ks, cta_pair=1)
    assert same(Y, Y1)


def test_tile_m_64_and_micro_batches(mc, oracle_mod):
    M, dims = 320, (1024, 768, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=83)
    Y, _, info = run_chain(mc, X, Ws, tile_k=128, tile_m=64, tile_n=[128, 64], k_split=[2, 2])
    assert info["tile_m"] == 64 and info["fill_k"] == [128, 128]
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))
    Ym, _, _ = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=64, tile_k=128, tile_m=64,
                         tile_n=[128, 64], k_split=[2, 2])
    assert same(Y, Ym)


def run_gated(mc, X, Ws, dims, **kw):
    with mc.Chain(X.shape[0], dims, gated=True, **kw) as ch:
        ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=DEV)
        Y = torch.full((X.shape[0], dims[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        ch.run(X.to(DEV), [w.to(DEV) for w in Ws], Y, ws)
        assert ch.check() == 0
        return Y.cpu(), ch.info()


def test_gated_chain_fills_its_down_projection_deep(mc, oracle_mod):
    M, dims = 256, (1024, 768, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims, gated=True), seed=84)
    Y, info = run_gated(mc, X, Ws, dims, tile_k=128, tile_n=[128, 128], k_split=[1, 2])
    assert info["fill_k"] == [64, 128]   # the gated GEMM's slot holds gate and up tiles: one block
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gated=True))
    Y1, _ = run_gated(mc, X, Ws, dims, tile_k=64, tile_n=[128, 128], k_split=[1, 2])
    assert same(Y, Y1)


def test_gelu_residual_four_gemms(mc, oracle_mod):
    M, dims = 256, (512, 1024, 768, 512, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims, gelu=True, residual=True), seed=85)
    kw = dict(gelu=True, residual=True, cta_pair=1, tile_n=[128] * 4, k_split=[1] * 4)
    Y, _, info = run_chain(mc, X, Ws, tile_k=128, **kw)
    assert info["fill_k"] == [128] * 4
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True))
    Y1, _, _ = run_chain(mc, X, Ws, tile_k=64, **kw)
    assert same(Y, Y1)


def test_integer_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(256, (1024, 768, 512), seed=86)
    Y, H, info = run_chain(mc, X, Ws, tile_k=128, tile_n=[128, 128], k_split=[2, 2], cta_pair=1)
    assert info["fill_k"] == [128, 128]
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_repeated_runs_are_identical(mc):
    X, Ws = si.draw(si.make_workload("t", 128, (2048, 1024, 1024)), seed=87)
    outs, _, _ = run_chain(mc, X, Ws, reps=3, tile_k=128, tile_n=[128, 128], k_split=[4, 4], cta_pair=1)
    assert same(outs[0], outs[1]) and same(outs[0], outs[2])
