"""GPU parity of the gated (SwiGLU) first stage through the C ABI: H = SiLU(X Wg) * (X Wu).

The gated stage issues two MMAs per k step (gate and up weights, one activation tile) into two
fp32 accumulators side by side in TMEM, and the epilogue rounds SiLU(gate) * up once.  Bar:
H and Y within |d| <= 1e-2 (|ref| + 1) of the oracle per element; every launch mode and both
weight layouts bit-identical.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from test_gpu_chain import DEV, assert_close_to_oracle, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mc():
    import mlp_latency_gb300
    mlp_latency_gb300.build()
    mlp_latency_gb300.load()
    return mlp_latency_gb300


def run_gated(mc, X, Ws, dims, mode="pipelined", reps=1, layout="kn", **kw):
    M = X.shape[0]
    Wd = [(w.t().contiguous() if layout == "nk" else w).to(DEV) for w in Ws]
    with mc.Chain(M, dims, mode=mode, gated=True, weight_layout=layout, **kw) as ch:
        ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=DEV)
        Y = torch.full((M, dims[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        outs = []
        for _ in range(reps):
            Y.fill_(float("nan"))
            ch.run(X.to(DEV), Wd, Y, ws)
            assert ch.check() == 0
            outs.append(Y.cpu().clone())
        H = ws[: M * dims[1] * 2].view(torch.bfloat16).view(M, dims[1]).cpu()
    return (outs if reps > 1 else outs[0]), H


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,dims,tn,ks", [
    (128, (256, 512, 256), [128, 64], None),
    (300, (512, 384, 512), [64, 128], [1, 2]),      # ragged rows, split-K in the second GEMM
    (200, (1000, 328, 96), None, None),             # ragged K and N, library tiles
    (64, (256, 256, 256), [32, 64], None),          # 32-wide gated tiles (64-byte swizzle)
])
def test_gated_matches_oracle_in_every_mode(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims, gated=True), seed=41)
    Y, H = run_gated(mc, X, Ws, dims, tile_n=tn, k_split=ks)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(w) for w in Ws], gated=True, return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    for mode, extra in (("sequential", {}), ("pipelined_kwait", {}), ("microbatch", {"microbatch_rows": 128})):
        if mode == "microbatch" and M <= 128:
            continue
        Ym, _ = run_gated(mc, X, Ws, dims, mode=mode, tile_n=tn, k_split=ks, **extra)
        assert same(Y, Ym), mode


def test_gated_weight_layouts_agree(mc):
    dims = (512, 256, 384)
    X, Ws = si.draw(si.make_workload("t", 256, dims, gated=True), seed=42)
    Ykn, _ = run_gated(mc, X, Ws, dims, tile_n=[128, 128])
    Ynk, _ = run_gated(mc, X, Ws, dims, layout="nk", tile_n=[128, 128])
    assert same(Ykn, Ynk)


def test_gated_three_stage_chain_with_gelu_after(mc, oracle_mod):
    # GeLU applies to the GEMMs after the gated one only
    dims = (256, 384, 256, 512)
    w = si.make_workload("t", 192, dims, gated=True, gelu=True)
    X, Ws = si.draw(w, seed=43)
    Y, _ = run_gated(mc, X, Ws, dims, gelu=True, tile_n=[64, 128, 64])
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws], gated=True, gelu=True))
    Ys, _ = run_gated(mc, X, Ws, dims, mode="sequential", gelu=True, tile_n=[64, 128, 64])
    assert same(Y, Ys)


def test_gated_zero_gate_gives_exact_zero(mc):
    # SiLU(0) = 0 exactly in the kernel too: a zero gate matrix zeroes H and Y bit for bit
    dims = (256, 256, 128)
    X, Ws = si.draw_integer(128, dims, seed=44, gated=True)
    Ws[0] = torch.zeros_like(Ws[0])
    Y, H = run_gated(mc, X, Ws, dims, tile_n=[128, 128])
    assert not torch.any(H.float() != 0) and not torch.any(Y.float() != 0)


def test_gated_repeated_runs_identical(mc):
    dims = (512, 512, 256)
    X, Ws = si.draw(si.make_workload("t", 256, dims, gated=True), seed=45)
    outs, _ = run_gated(mc, X, Ws, dims, reps=4, tile_n=[128, 64])
    for o in outs[1:]:
        assert same(o, outs[0])


def test_gated_llama_full_size_sampled_rows(mc, oracle_mod):
    w = si.WORKLOADS["llama_swiglu_m256_4096_14336"]
    X, Ws = si.draw(w, seed=0)
    Y, _ = run_gated(mc, X, Ws, w.dims)
    rows = si.sample_rows(w.M, 24, seed=5)
    Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws], gated=True, rows=rows)
    assert_close_to_oracle(Y[torch.as_tensor(rows)], Yo)
    Yk, _ = run_gated(mc, X, Ws, w.dims, mode="pipelined_kwait")
    assert same(Y, Yk)


@pytest.mark.parametrize("M,dims,tn,ks", [
    (256, (1024, 1536, 1024), [128, 256], [1, 4]),     # the down-projection's slices on separate clusters
    (200, (512, 640, 512), [64, 128], [1, 2]),         # 64-wide gated pair tiles, ragged rows
    (512, (1024, 1024, 512), [128, 128], [1, 1]),      # two pair panels
])
def test_gated_pairs_match_oracle_and_one_cta_tiles(mc, oracle_mod, M, dims, tn, ks):
    """On a CTA pair the leader loads the gate tile and the peer the up tile; the pair's MMA is as
    wide as both and each CTA's accumulator holds its rows of gate and up side by side.  Same bits
    as one CTA per tile."""
    X, Ws = si.draw(si.make_workload("t", M, dims, gated=True), seed=45)
    Yp, Hp = run_gated(mc, X, Ws, dims, tile_n=tn, k_split=ks, cta_pair=2)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(w) for w in Ws], gated=True, return_h=True)
    assert_close_to_oracle(Hp, Ho)
    assert_close_to_oracle(Yp, Yo)
    Y1, H1 = run_gated(mc, X, Ws, dims, tile_n=tn, k_split=ks, cta_pair=1)
    assert same(Yp, Y1) and same(Hp, H1)
    Ys, _ = run_gated(mc, X, Ws, dims, mode="sequential", tile_n=tn, k_split=ks, cta_pair=2)
    assert same(Yp, Ys)
    if M % 256 == 0 and M > 256:   # pair micro-batch chunks hold whole 256-row tiles
        Ym, _ = run_gated(mc, X, Ws, dims, mode="microbatch", microbatch_rows=256, tile_n=tn, k_split=ks, cta_pair=2)
        assert same(Yp, Ym)


def test_gated_llama_library_choice_sampled(mc, oracle_mod):
    """The SwiGLU Llama MLP with the library's plan (CTA pairs, the down-projection's slices on
    separate clusters where the model puts them ahead), on sampled rows, and the same bits as the
    sequential launches of the same tiles."""
    w = si.WORKLOADS["llama_swiglu_m256_4096_14336"]
    X, Ws = si.draw(w, seed=0)
    with mc.Chain(w.M, w.dims, gated=True) as ch:
        info = ch.info()
    Y, _ = run_gated(mc, X, Ws, w.dims)
    rows = si.sample_rows(w.M, 12, seed=5)
    assert_close_to_oracle(Y[rows], oracle_mod.chain(bits(X), [bits(t) for t in Ws], gated=True, rows=rows))
    Ys, _ = run_gated(mc, X, Ws, w.dims, mode="sequential", tile_n=info["tile_n"], k_split=info["k_split"],
                      cta_pair=info["cta_pair"])
    assert same(Y, Ys)
