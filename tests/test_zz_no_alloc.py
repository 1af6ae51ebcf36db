"""The allocation-free entry point, through the C ABI, against the regular entry point and the oracle.

mlp_chain_run_noalloc exists for callers that cannot allocate device memory while they run
the chain (allocator callbacks, runtimes that reserve all device memory up front, embeddings
that must bypass the framework's allocator); all of its scratch lives in one static device
array.  This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu
TOL = 1e-2
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    import mlp_latency_gb300
    mlp_latency_gb300.build()
    return mlp_latency_gb300.load()


def regular_entry_point(X, W1, W2, **kw):
    import mlp_latency_gb300 as mc
    M, dims = X.shape[0], (X.shape[1], W1.shape[1], W2.shape[1])
    with mc.Chain(M, dims, mode="pipelined", **kw) as ch:
        ws = torch.empty(ch.workspace_size(), dtype=torch.uint8, device=DEV)
        Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
        ch.run(X, [W1, W2], Y, ws)
        assert ch.check() == 0
    return Y


def noalloc(lib, X, W1, W2, Y, sync_check=1):
    st = torch.cuda.current_stream().cuda_stream or None
    return lib.mlp_chain_run_noalloc(X.shape[0], X.shape[1], W1.shape[1], W2.shape[1], X.data_ptr(),
                                     W1.data_ptr(), W2.data_ptr(), Y.data_ptr(), sync_check, st)


@pytest.mark.parametrize("M,dims", [(128, (4096, 4096, 4096)), (300, (512, 1024, 264))])
def test_noalloc_matches_regular_entry_point_twice(lib, M, dims):
    """Bit for bit against mlp_chain_run with the same tiles (unsplit, the library's tile widths),
    within tolerance of the default (split-K) handle, on two calls in a row."""
    X, (W1, W2) = si.draw(si.make_workload("t", M, dims), seed=21)
    Xd, W1d, W2d = X.to(DEV), W1.to(DEV), W2.to(DEV)
    same_tiles = regular_entry_point(Xd, W1d, W2d, k_split=[1, 1])
    default = regular_entry_point(Xd, W1d, W2d).float()
    for _ in range(2):   # the second call reuses the static scratch left by the first
        Y = torch.full((M, dims[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert noalloc(lib, Xd, W1d, W2d, Y) == 0
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), same_tiles.view(torch.int16))
        err = (Y.float() - default).abs()
        assert bool((err <= TOL * (default.abs() + 1)).all()), float(err.max())


def test_noalloc_matches_the_oracle(lib, oracle_mod):
    M, dims = 200, (320, 512, 264)    # two row panels, a ragged last one
    X, Ws = si.draw(si.make_workload("t", M, dims), seed=22)
    Xd, W1d, W2d = (t.to(DEV) for t in (X, *Ws))
    Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
    for _ in range(2):
        assert noalloc(lib, Xd, W1d, W2d, Y) == 0
        ref = oracle_mod.bf16_to_f32(oracle_mod.chain(si.bits(X), [si.bits(t) for t in Ws]))
        got = Y.float().cpu().numpy()
        assert np.all(np.abs(got - ref) <= TOL * (np.abs(ref) + 1))


def test_noalloc_takes_no_device_memory(lib):
    """After a warm-up call, further calls change neither the device's free memory nor torch's
    allocator."""
    M, dims = 256, (1024, 2048, 512)
    X, (W1, W2) = si.draw(si.make_workload("t", M, dims), seed=23)
    Xd, W1d, W2d = X.to(DEV), W1.to(DEV), W2.to(DEV)
    Y = torch.empty(M, dims[-1], dtype=torch.bfloat16, device=DEV)
    assert noalloc(lib, Xd, W1d, W2d, Y) == 0           # warm-up: module and kernel image loaded
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        assert noalloc(lib, Xd, W1d, W2d, Y, sync_check=0) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_rejects_shapes_beyond_the_static_scratch(lib):
    M, N1 = 2048, 8192                # H alone is 32 MiB > the 16 MiB array
    X = torch.zeros(M, 64, dtype=torch.bfloat16, device=DEV)
    W1 = torch.zeros(64, N1, dtype=torch.bfloat16, device=DEV)
    W2 = torch.zeros(N1, 64, dtype=torch.bfloat16, device=DEV)
    Y = torch.zeros(M, 64, dtype=torch.bfloat16, device=DEV)
    assert noalloc(lib, X, W1, W2, Y) == 1   # MLP_ERR_INVALID_ARG, nothing enqueued
