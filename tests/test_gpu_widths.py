"""GPU parity of tile widths that are not powers of two (multiples of 32 up to 256).

Such a tile's last 64-column box of weights is loaded whole (the columns past the tile are
read and not used; past N they are zero-filled), with one 2-D copy per box; the MMA's N is the
tile width.  Bar: within |d| <= 1e-2 (|ref| + 1) of the oracle; bit-identical between CTA pairs
and one CTA per tile, and across launch modes, at the same widths and splits.
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
    (512, (512, 1120, 672), [224, 224]),     # whole tiles
    (300, (448, 704, 520), [224, 160]),      # ragged rows and columns: the last tile's boxes run past N
    (640, (1024, 576, 384), [192, 192]),
])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_pairs_at_odd_widths_match_oracle_and_one_cta_tiles(mc, oracle_mod, M, dims, tn, layout):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=71)
    Wl = [w.t().contiguous() for w in Ws] if layout == "nk" else Ws
    Yp, Hp, info = run_chain(mc, X, Wl, tile_n=tn, k_split=[1, 1], cta_pair=2, weight_layout=layout)
    assert info["tile_n"] == tn and info["cta_pair"] == 2
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(Hp, Ho)
    assert_close_to_oracle(Yp, Yo)
    Ys, Hs, info1 = run_chain(mc, X, Wl, tile_n=tn, k_split=[1, 1], cta_pair=1, weight_layout=layout)
    assert info1["cta_pair"] == 1
    assert same(Hp, Hs) and same(Yp, Ys)
    for mode in ("sequential", "sequential_pdl"):
        Y, _, _ = run_chain(mc, X, Wl, mode=mode, tile_n=tn, k_split=[1, 1], cta_pair=2, weight_layout=layout)
        assert same(Yp, Y), mode


@pytest.mark.parametrize("tn,ks", [([96, 160], [1, 1]), ([192, 224], [2, 1]), ([224, 192], [1, 2])])
def test_one_cta_odd_widths_and_split_k(mc, oracle_mod, tn, ks):
    M, dims = 257, (1024, 448, 768)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=72)
    Y, H, info = run_chain(mc, X, Ws, tile_n=tn, k_split=ks, cta_pair=1)
    assert info["tile_n"] == tn and info["k_split"] == ks
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=ks, cta_pair=1)
    assert same(Y, Ys)
    Ym, _, _ = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=128, tile_n=tn, k_split=ks, cta_pair=1)
    assert same(Y, Ym)


def test_pair_split_k_at_192(mc, oracle_mod):
    M, dims = 512, (2048, 576, 384)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=73)
    Yp, _, info = run_chain(mc, X, Ws, tile_n=[192, 192], k_split=[2, 2], cta_pair=2)
    assert info["cluster_size"] == 4
    Ys, _, _ = run_chain(mc, X, Ws, tile_n=[192, 192], k_split=[2, 2], cta_pair=1)
    assert same(Yp, Ys)
    assert_close_to_oracle(Yp, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_integer_inputs_are_bit_exact_at_224(mc, oracle_mod):
    X, Ws = si.draw_integer(512, (1024, 896, 448), seed=74)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[224, 224], cta_pair=2, k_split=[1, 1])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_widths_refused(mc):
    """Widths must be multiples of 32, a split must leave 32-column multiples per owner, and a
    gated GEMM takes 32, 64 or 128."""
    for kw in (dict(tile_n=[100, 128]), dict(tile_n=[224, 224], k_split=[2, 1]),
               dict(tile_n=[96, 128], gated=True)):
        dims = (512, 512, 512)
        with pytest.raises(mc.MlpChainError) as e:
            mc.Chain(256, dims, **kw)
        assert e.value.status == mc.ERR_UNSUPPORTED, kw


def test_gelu_chain_odd_width_pairs_sampled(mc, oracle_mod):
    """The 4-GEMM GeLU chain at its full size with 224-wide pair tiles (74 tiles on 76 pairs)."""
    w = si.WORKLOADS["gelu4_m512_d8192"]
    X, Ws = si.draw(w, seed=0)
    Y, _, info = run_chain(mc, X, Ws, gelu=True, residual=True, tile_n=[224] * 4, k_split=[1] * 4, cta_pair=2)
    rows = si.sample_rows(w.M, 12, seed=8)
    assert_close_to_oracle(Y[rows], oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True, rows=rows))
