"""GPU tests of mlp_chain_run_host, the entry point with HOST input and output buffers.

X is copied from the host into the device staging buffer; the result reaches Y_host either
through the last GEMM's epilogue storing straight into page-locked host memory, or (pageable
Y_host) through the device buffer Y_dev and a copy.  Both give the bits of mlp_chain_run.
"""
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


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("mode", ["pipelined", "sequential", "microbatch"])
@pytest.mark.parametrize("pinned", [True, False])
def test_run_host_matches_device_run(mc, oracle_mod, mode, pinned):
    M, dims = 384, (512, 768, 256)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=61)
    Wd = [w.to(DEV) for w in Ws]
    kw = dict(microbatch_rows=128) if mode == "microbatch" else {}
    with mc.Chain(M, dims, mode=mode, **kw) as ch:
        ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(X.to(DEV), Wd, Y, ws)
        assert ch.check() == 0
        Xh = X.pin_memory() if pinned else X.clone()
        Yh = torch.full((M, dims[-1]), float("nan"), dtype=torch.bfloat16)
        if pinned:
            Yh = Yh.pin_memory()
        Xs = torch.empty_like(Y.new_empty(M, dims[0]))
        Yd = torch.full((M, dims[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        for _ in range(2):
            ch.run_host(Xh, Wd, Yh, Xs, Yd, ws)
            assert ch.check() == 0
            assert same(Yh, Y.cpu())
        # page-locked output is written by the epilogue directly; the device buffer stays untouched
        assert bool(torch.isnan(Yd.float()).all()) == pinned
    assert_close_to_oracle(Yh, oracle_mod.chain(bits(X), [bits(t) for t in Ws]))


def test_run_host_pairs_and_split_k(mc):
    """The direct store path under CTA pairs with split-K (the global-memory exchange ends in the
    owners' stores of their slices)."""
    M, dims = 512, (2048, 512, 1024)
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=62)
    Wd = [w.to(DEV) for w in Ws]
    with mc.Chain(M, dims, tile_n=[256, 256], k_split=[2, 4], cta_pair=2) as ch:
        ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(X.to(DEV), Wd, Y, ws)
        assert ch.check() == 0
        Yh = torch.empty(M, dims[-1], dtype=torch.bfloat16).pin_memory()
        Xs = torch.empty(M, dims[0], dtype=torch.bfloat16, device=DEV)
        Yd = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run_host(X.pin_memory(), Wd, Yh, Xs, Yd, ws)
        assert ch.check() == 0
        assert same(Yh, Y.cpu())
