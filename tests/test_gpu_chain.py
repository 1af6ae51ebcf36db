"""GPU parity of the CUDA chain (through the C ABI) against the CPU oracle.

Bar: Y within |d| <= 1e-2 (|ref| + 1) per element of the oracle; bit-exact on integer-valued
inputs and closed forms; bit-identical across the pipelined, sequential and micro-batched
launch modes (same tiles, same k order); the event log shows no consumer tile starting before
all of its producer tiles finished.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def mc():
    import mlp_latency_gb300
    mlp_latency_gb300.build()
    mlp_latency_gb300.load()
    return mlp_latency_gb300


DEV = torch.device("cuda:0")


def run_chain(mc, X, Ws, mode="pipelined", reps=1, **kw):
    col = 0 if kw.get("weight_layout") == "nk" else 1
    M, dims = X.shape[0], [X.shape[1]] + [w.shape[col] for w in Ws]
    Xd = X.to(DEV)
    Wd = [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, mode=mode, **kw) as ch:
        ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=DEV)
        Y = torch.full((M, dims[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        outs = []
        for _ in range(reps):
            Y.fill_(float("nan"))
            ch.run(Xd, Wd, Y, ws)
            st = ch.check()
            assert st == 0, f"device status {st}"
            outs.append(Y.cpu().clone())
        H = ws[: M * dims[1] * 2].view(torch.bfloat16).view(M, dims[1]).cpu() if len(Ws) > 1 else None
        info = ch.info()
    return outs if reps > 1 else outs[0], H, info


def assert_close_to_oracle(got, ref_bits):
    ref = (ref_bits.astype(np.uint32) << 16).view(np.float32)
    g = got.float().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= TOL * (np.abs(ref) + 1))
    assert not bad.any(), (f"{int(bad.sum())}/{bad.size} outside tolerance; worst {float(err.max())} "
                           f"at {np.unravel_index(np.argmax(err), err.shape)}")


def bits(t):
    return si.bits(t)


# ----------------------------------------------------------------------------- tiny chain --
def test_tiny_pipelined_matches_oracle(mc, oracle_mod):
    w = si.WORKLOADS["tiny_m64_d256"]
    X, Ws = si.draw(w, seed=0)
    Y, H, info = run_chain(mc, X, Ws, tile_n=[64, 64])
    assert info["tiles_n"] == [4, 4] and info["launches_per_run"] == 1
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
def test_every_tile_width_matches_oracle(mc, oracle_mod, bn):
    w = si.make_workload("t", 200, (320, 512, 264))
    X, Ws = si.draw(w, seed=1)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[bn, bn])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)


@pytest.mark.parametrize("M,dims", [(1, (64, 64, 64)), (130, (72, 136, 40)), (257, (1000, 328, 96)),
                                    (384, (128, 2048, 128))])
def test_ragged_shapes_match_oracle(mc, oracle_mod, M, dims):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=2)
    Y, H, _ = run_chain(mc, X, Ws)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)


def test_integer_valued_inputs_are_bit_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(300, (1024, 1024, 512), seed=11)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[128, 64])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_identity_and_permutation_closed_forms(mc):
    M, d = 192, 256
    X, _ = si.draw(si.make_workload("t", M, (d, d, d)), seed=7)
    I = torch.eye(d, dtype=torch.bfloat16)
    P, perm = si.permutation_matrix(d, seed=3)
    Y, _, _ = run_chain(mc, X, [I, P], tile_n=[64, 128])
    expect = torch.empty_like(X)
    expect[:, perm] = X
    assert torch.equal(Y.view(torch.int16), expect.view(torch.int16))


# ------------------------------------------------------------------------------ the modes --
@pytest.mark.parametrize("M,dims,tn", [(512, (512, 1024, 256), [128, 64]), (300, (256, 384, 512), [64, 128]),
                                       (1024, (256, 256, 256), [256, 32])])
def test_modes_are_bit_identical(mc, M, dims, tn):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=4)
    Yp, _, _ = run_chain(mc, X, Ws, tile_n=tn)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn)
    assert torch.equal(Yp.view(torch.int16), Ys.view(torch.int16))
    for rows in (128, 256):
        if rows < M:
            Ym, _, info = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=rows, tile_n=tn)
            assert info["launches_per_run"] == 2 * -(-M // rows)
            assert torch.equal(Yp.view(torch.int16), Ym.view(torch.int16))


def test_repeated_runs_of_one_handle_are_identical(mc):
    X, Ws = si.draw(si.make_workload("t", 640, (256, 512, 256)), seed=6)
    outs, _, _ = run_chain(mc, X, Ws, reps=5, tile_n=[64, 64])
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("grid,ks,tn", [(3, [1, 1], [64, 64]), (4, [2, 2], [64, 64]), (8, [4, 1], [128, 64])])
def test_small_grid_still_completes(mc, oracle_mod, grid, ks, tn):
    # fewer CTAs than tiles: every cluster loops over producer and consumer tickets
    X, Ws = si.draw(si.make_workload("t", 512, (256, 512, 256)), seed=8)
    Y, _, info = run_chain(mc, X, Ws, tile_n=tn, grid_ctas=grid, k_split=ks)
    assert info["grid_ctas"] == grid
    assert_close_to_oracle(Y, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_grouped_raster_matches(mc):
    X, Ws = si.draw(si.make_workload("t", 1024, (256, 512, 256)), seed=9)
    Ya, _, _ = run_chain(mc, X, Ws, tile_n=[64, 64])
    Yb, _, _ = run_chain(mc, X, Ws, tile_n=[64, 64], raster_group=3)
    assert torch.equal(Ya.view(torch.int16), Yb.view(torch.int16))


# ------------------------------------------------------------------------ the protocol log --
# 640 rows: one scoreboard group per row panel; 1152 rows (9 panels): groups merged per raster
# group of 4 (4, 4, 1 panels) or 3, consumers pushed column by column
@pytest.mark.parametrize("M,rg", [(640, 0), (1152, 0), (1152, 3)])
def test_event_log_respects_every_dependency(mc, oracle_mod, M, rg):
    dims, tn = (256, 512, 384), [64, 128]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=10)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, event_log=True, raster_group=rg) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        for _ in range(2):   # the second run checks the re-armed scoreboard
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
            log = ch.event_log()
            off, tgt, init = ch.deps(0)
            info = ch.info()
            P = info["tiles_m"][0] * info["tiles_n"][0]
            C = info["tiles_m"][1] * info["tiles_n"][1]
            assert len(log) == P + C
            prod, cons = log[:P], log[P:]
            assert np.array_equal(prod["stage"], np.zeros(P)) and np.array_equal(prod["tile"], np.arange(P))
            assert np.array_equal(cons["stage"], np.ones(C)) and np.array_equal(cons["tile"], np.arange(C))
            seqs = np.concatenate([log["seq_start"], log["seq_end"][:P]])
            assert len(set(seqs.tolist())) == len(seqs)
            for p in range(P):
                for c in tgt[off[p]:off[p + 1]]:
                    assert prod["seq_end"][p] < cons["seq_start"][c]
                    assert prod["t_end"][p] <= cons["t_start"][c]
            assert np.all(init == info["tiles_n"][0])
        Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws])
        assert_close_to_oracle(Y.cpu(), Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn)
    assert torch.equal(Y.cpu().view(torch.int16), Ys.view(torch.int16))


@pytest.mark.parametrize("M,grid,queue_free", [
    (256, 0, 1),    # two scoreboard groups, a cluster for every consumer: no queue
    (256, 4, 0),    # two groups, 8 consumer tiles on 4 CTAs: the queue
    (128, 0, 1),    # one group: no queue
])
def test_dropped_decrement_times_out_then_recovers(mc, M, grid, queue_free):
    dims = (256, 256, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=12)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=[64, 64], k_split=[1, 1], drop_tile=1, timeout_us=20000, grid_ctas=grid,
                  raster_group=1) as ch:
        assert ch.info()["queue_free"] == [queue_free]
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)                    # tile 1 withholds its decrements
        assert ch.check() == mc.ERR_TIMEOUT      # ... so its consumers' bounded wait ran out
        ch.run(Xd, Wd, Y, ws)                    # the fault fires once; check() re-armed the handle
        assert ch.check() == 0
        Y2 = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=[64, 64], k_split=[1, 1])
    assert torch.equal(Y2.view(torch.int16), Ys.view(torch.int16))


def test_invalid_pointers_are_rejected(mc):
    with mc.Chain(128, (256, 256, 256)) as ch:
        X = torch.zeros(128, 256, dtype=torch.bfloat16, device=DEV)
        W = [torch.zeros(256, 256, dtype=torch.bfloat16, device=DEV)] * 2
        Y = torch.zeros(128, 256, dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(ch.workspace_size() + 512, dtype=torch.uint8, device=DEV)
        with pytest.raises(mc.MlpChainError):
            ch.run(X, W, Y, None)
        with pytest.raises(mc.MlpChainError):
            ch.run(X.view(-1)[1:], W, Y, ws)          # misaligned X
        with pytest.raises(mc.MlpChainError):
            ch.run(X, W, Y, ws[16:])                  # misaligned workspace


# ---------------------------------------------------------------------- GeLU + residual --
def test_gelu_residual_four_gemm_chain(mc, oracle_mod):
    w = si.make_workload("t", 300, (512,) * 5, gelu=True, residual=True)
    X, Ws = si.draw(w, seed=14)
    Y, _, _ = run_chain(mc, X, Ws, gelu=True, residual=True, tile_n=[64, 128, 64, 128])
    Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=True, residual=True)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", gelu=True, residual=True, tile_n=[64, 128, 64, 128])
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16))
    Ym, _, _ = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=128, gelu=True, residual=True,
                         tile_n=[64, 128, 64, 128])
    assert torch.equal(Y.view(torch.int16), Ym.view(torch.int16))


# ------------------------------------------------------------------ full-size workloads --
@pytest.mark.parametrize("name", ["decode_m128_d4096", "llama_m256_4096_14336", "prefill_m2048_d8192",
                                  "gelu4_m512_d8192"])
def test_full_size_workloads_sampled_rows(mc, oracle_mod, name):
    w = si.WORKLOADS[name]
    X, Ws = si.draw(w, seed=0)
    Y, _, info = run_chain(mc, X, Ws, gelu=w.gelu, residual=w.residual)
    rows = si.sample_rows(w.M, 32, seed=1)
    Yo = oracle_mod.chain(bits(X), [bits(t) for t in Ws], gelu=w.gelu, residual=w.residual, rows=rows)
    assert_close_to_oracle(Y[torch.from_numpy(rows)], Yo)
    # properties that hold at any size: every element finite and written
    assert torch.isfinite(Y.float()).all()


# --------------------------------------------------------------------- tuning knobs --
@pytest.mark.parametrize("bn,split,stages", [(32, 2, 0), (128, 2, 3), (64, 1, 2), (256, 1, 2)])
def test_split_accumulators_and_ring_depth(mc, oracle_mod, bn, split, stages):
    X, Ws = si.draw(si.make_workload("t", 384, (1024, 512, 320)), seed=15)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[bn, bn], acc_split=split, pipe_stages=stages)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=[bn, bn], acc_split=split, pipe_stages=stages)
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16))


def test_split_accumulators_integer_inputs_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(200, (1024, 512, 256), seed=16)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[64, 32], acc_split=2)
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
def test_transposed_weight_layout(mc, oracle_mod, bn):
    # weights stored N x K (nn.Linear layout): B is K-major in shared memory
    X, Ws = si.draw(si.make_workload("t", 272, (640, 384, 264)), seed=17)
    Wt = [w.t().contiguous() for w in Ws]
    Y, H, _ = run_chain(mc, X, Wt, tile_n=[bn, bn], weight_layout="nk")
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Wt, mode="sequential", tile_n=[bn, bn], weight_layout="nk")
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16))


# --------------------------------------------------------------------------- split-K --
@pytest.mark.parametrize("M,dims,tn,ks", [
    (128, (2048, 1024, 2048), [256, 256], [8, 8]),
    (300, (1024, 512, 384), [128, 64], [4, 2]),
    (200, (512, 768, 256), [256, 256], [2, 1]),
    (128, (4096, 512, 256), [64, 32], [2, 1]),
    (257, (1000, 328, 96), None, None),          # library choice: mixed splits in one cluster
])
def test_split_k_matches_oracle_and_modes(mc, oracle_mod, M, dims, tn, ks):
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=18)
    Y, H, info = run_chain(mc, X, Ws, tile_n=tn, k_split=ks)
    if ks:
        assert info["k_split"] == ks and info["cluster_size"] == max(ks) * info["cta_pair"]
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert_close_to_oracle(H, Ho)
    assert_close_to_oracle(Y, Yo)
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=ks)
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16))
    if ks and max(tn) <= 128:   # the shared-memory exchange adds the same parts in the same order
        Yd, Hd, _ = run_chain(mc, X, Ws, tile_n=tn, k_split=ks, splitk_exchange="dsmem")
        assert torch.equal(Y.view(torch.int16), Yd.view(torch.int16))
        assert torch.equal(H.view(torch.int16), Hd.view(torch.int16))
    if M > 128:
        Ym, _, _ = run_chain(mc, X, Ws, mode="microbatch", microbatch_rows=128, tile_n=tn, k_split=ks)
        assert torch.equal(Y.view(torch.int16), Ym.view(torch.int16))


def test_split_k_integer_inputs_exact(mc, oracle_mod):
    X, Ws = si.draw_integer(256, (2048, 512, 1024), seed=19)
    Y, H, _ = run_chain(mc, X, Ws, tile_n=[128, 256], k_split=[4, 8])
    Yo, Ho = oracle_mod.chain(bits(X), [bits(t) for t in Ws], return_h=True)
    assert np.array_equal(bits(H), Ho)
    assert np.array_equal(bits(Y), Yo)


def test_split_k_event_log_and_repeat(mc):
    M, dims, tn, ks = 384, (2048, 1024, 512), [256, 128], [4, 2]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=20)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, k_split=ks, event_log=True) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        first = None
        for _ in range(3):
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
            if first is None:
                first = Y.clone()
            assert torch.equal(Y.view(torch.int16), first.view(torch.int16))
            log = ch.event_log()
            off, tgt, _ = ch.deps(0)
            P = len(off) - 1
            prod, cons = log[:P], log[P:]
            assert np.array_equal(prod["tile"], np.arange(P)) and np.array_equal(cons["tile"], np.arange(len(cons)))
            for p in range(P):
                for c in tgt[off[p]:off[p + 1]]:
                    assert prod["seq_end"][p] < cons["seq_start"][c]


def test_split_k_dropped_decrement_times_out_then_recovers(mc):
    M, dims = 256, (1024, 512, 512)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=22)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=[128, 128], k_split=[4, 2], drop_tile=0, timeout_us=20000) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == mc.ERR_TIMEOUT
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == 0
        Y2 = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=[128, 128], k_split=[4, 2])
    assert torch.equal(Y2.view(torch.int16), Ys.view(torch.int16))


# ------------------------------------------------------------------------- the scoreboard --
@pytest.mark.parametrize("M,dims,tn,ks,rg", [
    (128, (4096, 4096, 4096), [128, 128], [4, 4], 0),        # decode: one group, split releases
    (2048, (1024, 1024, 512), [256, 128], [1, 1], 0),        # 16 panels: merged groups of 8
    (1152, (512, 768, 256), [128, 64], [1, 2], 3),           # 9 panels, groups of 3, split consumer
    (300, (256, 384, 512), [64, 128], [1, 1], 1),            # ragged, unmerged
    (512, (512, 512, 512, 512, 512), [128, 128, 128, 128], [1, 1, 1, 1], 0),   # 3 boundaries
])
@pytest.mark.parametrize("cp", [1, 0])   # one CTA per tile, and the library's choice (pairs where they apply)
def test_device_scoreboard_matches_oracle_enumeration(mc, oracle_mod, M, dims, tn, ks, rg, cp):
    """The counters' tables as the kernel reads them (copied back from the device) equal the ones
    rebuilt from the oracle's brute-force enumeration, bit for bit, for every stage boundary."""
    import expected_scoreboard as es
    with mc.Chain(M, dims, tile_n=tn, k_split=ks, raster_group=rg, cta_pair=cp) as ch:
        info = ch.info()
        tiles_m = info["tiles_m"][0]
        g = info["raster_group"]
        assert (g == rg) if rg else (g == 8 if tiles_m >= 16 else g == 4 if tiles_m >= 8 else g in (1, tiles_m))
        for b in range(len(dims) - 2):
            # releases per producer tile: each epilogue warp of each of its CTAs (split-K slices x pair)
            rel = info["cta_pair"] * info["k_split"][b] * 4
            want = es.expected(oracle_mod, M, dims[b + 1], dims[b + 2], info["tile_m"], info["tile_n"][b],
                               info["tile_n"][b + 1], g, rel)
            es.assert_equal(ch.scoreboard(b), want)


def test_cta_lifetime_records_bracket_every_tile(mc):
    """The per-CTA records of the event log (entry, set-up done, exit) are ordered and enclose the
    start and release of every tile."""
    M, dims = 512, (256, 512, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=12)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=[64, 64], event_log=True) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(Xd, Wd, Y, ws)
        assert ch.check() == 0
        ctas, tiles, grid = ch.cta_log(), ch.event_log(), ch.info()["grid_ctas"]
    assert len(ctas) == grid and sorted(ctas["cta"].tolist()) == list(range(grid))
    assert (ctas["stage"] == -1).all()
    assert (ctas["t_start"] <= ctas["t_acc"]).all() and (ctas["t_acc"] <= ctas["t_end"]).all()
    assert tiles["t_start"].min() >= ctas["t_acc"].min() and tiles["t_end"].max() <= ctas["t_end"].max()


@pytest.mark.parametrize("mode", ["pipelined", "pipelined_kwait", "pipelined_lamport"])
def test_many_runs_of_one_handle_without_any_reset(mc, mode):
    """Tickets, queue tails, scoreboard counters and the launch counter accumulate over runs and
    are read relative to each run's epoch: forty back-to-back runs (split-K releases, merged
    scoreboard groups, a partial last row panel) all give the same bits."""
    M, dims = 1100, (256, 512, 384)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=13)
    outs, _, _ = run_chain(mc, X, Ws, mode=mode, reps=40, tile_n=[64, 128], k_split=[2, 2], raster_group=3)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_dsmem_exchange_rejects_tiles_wider_than_its_buffer(mc):
    """The shared-memory exchange holds S parts of a 128-row slice in 64 KB: 256-wide split tiles
    of 128 rows do not fit and are refused rather than silently sent through global memory."""
    with pytest.raises(mc.MlpChainError) as e:
        mc.Chain(256, (1024, 512, 512), tile_n=[256, 256], k_split=[2, 2], splitk_exchange="dsmem")
    assert e.value.status == mc.ERR_UNSUPPORTED
    with mc.Chain(256, (1024, 512, 512), tile_n=[256, 256], k_split=[2, 2]) as ch:
        assert ch.info()["k_split"] == [2, 2]


def test_library_raster_group_choice(mc):
    """Below 8 row panels the library groups all panels when the first stage takes more than one
    wave of cluster items, and none otherwise; from 8 panels up, groups of 4, then 8."""
    with mc.Chain(256, (4096, 14336, 4096), gated=True, cta_pair=1) as ch:   # SwiGLU MLP: 224 tiles, 36 clusters of 4
        assert ch.info()["raster_group"] == 2
    with mc.Chain(256, (4096, 14336, 4096)) as ch:               # Llama MLP: 112 tiles in one wave
        assert ch.info()["raster_group"] == 1
    with mc.Chain(1024, (8192, 8192, 8192)) as ch:               # 4 pair panels, 128 pair tiles on 76 pairs
        info = ch.info()
        assert info["cta_pair"] == 2 and info["raster_group"] == 4
    with mc.Chain(4096, (1024, 1024, 1024), cta_pair=1) as ch:    # 32 panels
        assert ch.info()["raster_group"] == 8
    with mc.Chain(4096, (1024, 1024, 1024), cta_pair=1, raster_group=3) as ch:
        assert ch.info()["raster_group"] == 3


@pytest.mark.parametrize("ks", [[1, 1], [2, 4]])
def test_single_group_boundary_skips_the_queue(mc, oracle_mod, ks):
    """One row panel: every consumer waits on the same group, so consumer slot q takes member q
    and acquires the counter directly.  Every dependency is still respected (event log, two runs)
    and Y matches the sequential launches bit for bit and the oracle within tolerance."""
    M, dims, tn = 128, (1024, 1024, 512), [128, 128]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=19)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, k_split=ks, event_log=True, cta_pair=1) as ch:
        assert ch.scoreboard(0)["groups"] == 1 and ch.info()["queue_free"] == [1]
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        for _ in range(2):
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
            ev = ch.event_log()
            off, tgt, _ = ch.deps(0)
            p_end = {int(e["tile"]): int(e["seq_end"]) for e in ev if e["stage"] == 0}
            c_start = {int(e["tile"]): int(e["seq_start"]) for e in ev if e["stage"] == 1}
            assert len(c_start) == 4
            for p in range(len(off) - 1):
                for c in tgt[off[p]:off[p + 1]]:
                    assert p_end[p] < c_start[int(c)]
        Yp = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=ks)
    assert torch.equal(Yp.view(torch.int16), Ys.view(torch.int16))
    assert_close_to_oracle(Yp, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


@pytest.mark.parametrize("grid,queue_free", [(0, 1), (8, 0)])
def test_one_wave_boundary_of_several_groups_skips_the_queue(mc, oracle_mod, grid, queue_free):
    """Four row panels (four scoreboard groups) and 16 consumer tiles: with a cluster for every
    consumer item the consumers take the groups' members in group order and acquire their group's
    counter (no queue); on 8 CTAs they poll the queue.  Both respect every dependency (event log,
    two runs) and give the sequential launches' bits."""
    M, dims, tn = 512, (1024, 1024, 512), [128, 128]
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=20)
    Xd, Wd = X.to(DEV), [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=tn, k_split=[1, 1], event_log=True, cta_pair=1, grid_ctas=grid,
                  raster_group=1) as ch:
        assert ch.scoreboard(0)["groups"] == 4 and ch.info()["queue_free"] == [queue_free]
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        for _ in range(2):
            ch.run(Xd, Wd, Y, ws)
            assert ch.check() == 0
            ev = ch.event_log()
            off, tgt, _ = ch.deps(0)
            p_end = {int(e["tile"]): int(e["seq_end"]) for e in ev if e["stage"] == 0}
            c_start = {int(e["tile"]): int(e["seq_start"]) for e in ev if e["stage"] == 1}
            assert len(p_end) == 32 and len(c_start) == 16
            for p in range(len(off) - 1):
                for c in tgt[off[p]:off[p + 1]]:
                    assert p_end[p] < c_start[int(c)]
        Yp = Y.cpu()
    Ys, _, _ = run_chain(mc, X, Ws, mode="sequential", tile_n=tn, k_split=[1, 1])
    assert torch.equal(Yp.view(torch.int16), Ys.view(torch.int16))
    assert_close_to_oracle(Yp, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))
