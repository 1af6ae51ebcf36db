"""Pins for the CPU oracle: each check rests on something other than the oracle itself.

* bf16 rounding    -- torch's own float32 -> bfloat16 cast, and hand-made ties.
* GeLU (tanh form) -- gelu(0) = 0, gelu(x) - gelu(-x) = x, limits, and torch's tanh-GeLU.
* GEMM chain       -- an exact (math.fsum, float64) triple loop on tiny shapes with the fp32
                      summation error bound; exact int64 results on integer-valued inputs;
                      identity / permutation / power-of-two closed forms.
* dependency array -- the tiny two-layer case worked by hand (golden file), the interval-overlap
                      closed form of the in-degree, and CSR invariants.
Planted mistakes (a transposed weight, a dropped term, a flipped sign) are shown to fail the pins.
"""
import math
import os

import numpy as np
import pytest
import torch

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------------- bf16 ----
def test_round_bf16_matches_torch(oracle_mod):
    rng = np.random.default_rng(1)
    scaled = rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)
    x = np.concatenate([
        scaled.astype(np.float32),
        rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-45, -1e-45], dtype=np.float32),
    ])
    ours = oracle_mod.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(f32(ours[nan])))


def test_round_bf16_ties_to_even(oracle_mod):
    one_plus_half_ulp = np.float32(1.0 + 2.0 ** -8)      # halfway between 1 and 1 + 2^-7
    three_halves = np.float32(1.0 + 3 * 2.0 ** -8)        # halfway between 1+2^-7 and 1+2^-6
    out = f32(oracle_mod.round_bf16(np.array([one_plus_half_ulp, three_halves, -one_plus_half_ulp])))
    assert out[0] == 1.0
    assert out[1] == 1.0 + 2.0 ** -6
    assert out[2] == -1.0


# ---------------------------------------------------------------------------------- GeLU ----
def test_gelu_identities(oracle_mod):
    assert oracle_mod.gelu(0.0) == 0.0
    for x in np.linspace(-6, 6, 97):
        g, gm = oracle_mod.gelu(x), oracle_mod.gelu(-x)
        assert abs((g - gm) - x) <= 1e-14 * max(1.0, abs(x))
    assert abs(oracle_mod.gelu(30.0) - 30.0) < 1e-12
    assert abs(oracle_mod.gelu(-30.0)) < 1e-12
    xs = np.linspace(0.0, 8.0, 200)
    assert all(oracle_mod.gelu(a) < oracle_mod.gelu(b) for a, b in zip(xs[:-1], xs[1:]))


def test_gelu_matches_torch_float64(oracle_mod):
    xs = torch.linspace(-8, 8, 1001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(xs, approximate="tanh")
    ours = torch.tensor([oracle_mod.gelu(float(v)) for v in xs], dtype=torch.float64)
    assert torch.max(torch.abs(ours - ref)).item() < 1e-13


def test_silu_identities(oracle_mod):
    # x*sigmoid(x): odd part x/2 (so silu(x) - silu(-x) = x), limits x and 0, and the textbook
    # minimum of about -0.27846 at x = -1.27846 (the root of 1 + x(1 - sigmoid(x)) = 0)
    assert oracle_mod.silu(0.0) == 0.0
    for x in np.linspace(-8, 8, 129):
        assert abs((oracle_mod.silu(x) - oracle_mod.silu(-x)) - x) <= 1e-14 * max(1.0, abs(x))
    assert abs(oracle_mod.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle_mod.silu(-40.0)) < 1e-12
    xs = np.linspace(-1.35, -1.2, 3001)
    vals = np.array([oracle_mod.silu(v) for v in xs])
    assert abs(xs[np.argmin(vals)] + 1.27846) < 1e-4 and abs(vals.min() + 0.27846) < 1e-5


def test_silu_matches_torch_float64(oracle_mod):
    xs = torch.linspace(-20, 20, 2001, dtype=torch.float64)
    ref = torch.nn.functional.silu(xs)
    ours = torch.tensor([oracle_mod.silu(float(v)) for v in xs], dtype=torch.float64)
    assert torch.max(torch.abs(ours - ref) / (1.0 + torch.abs(ref))).item() < 1e-15


def gated_bound_ok(got_bits, x, wg, wu):
    """H = SiLU(x wg) * (x wu) against the exact products (math.fsum) and an independent sigmoid
    (1 + tanh(z/2)) / 2.  Each fp32 accumulator is within g A of its exact value (any order of K
    additions); SiLU has slope below 1.1, so the product is within the linearised bound below,
    plus half a bf16 ulp of rounding."""
    K = x.shape[1]
    u = 2.0 ** -24
    g = K * u / (1 - K * u)
    ge, ue = exact_matmul(x, wg), exact_matmul(x, wu)
    dg = g * (np.abs(x.astype(np.float64)) @ np.abs(wg.astype(np.float64)))
    du = g * (np.abs(x.astype(np.float64)) @ np.abs(wu.astype(np.float64)))
    silu = ge * 0.5 * (1.0 + np.tanh(ge / 2.0))
    exact = silu * ue
    lin = 1.1 * dg * (np.abs(ue) + du) + np.abs(silu) * du + 1e-300
    bound = 2.0 ** -8 * (np.abs(exact) + lin) + lin * (1 + 1e-6)
    got = f32(got_bits).astype(np.float64)
    return bool(np.all(np.abs(got - exact) <= bound)), float(np.max(np.abs(got - exact) - bound))


@pytest.mark.parametrize("M,K,N1,N2", [(12, 32, 24, 40), (9, 64, 48, 16)])
def test_gated_chain_vs_exact_triple_loop(oracle_mod, M, K, N1, N2):
    w = si.make_workload("t", M, (K, N1, N2), gated=True)
    X, (Wg, Wu, W2) = si.draw(w, seed=5)
    Y, H = oracle_mod.chain(si.bits(X), [si.bits(Wg), si.bits(Wu), si.bits(W2)], gated=True,
                            return_h=True, threads=2)
    x, wg, wu, w2 = (f32(si.bits(t)) for t in (X, Wg, Wu, W2))
    ok, excess = gated_bound_ok(H, x, wg, wu)
    assert ok, excess
    ok, excess = stage_bound_ok(Y, f32(H), w2)     # the second stage is a plain GEMM of H
    assert ok, excess


def test_gated_chain_planted_mistakes_fail_the_pin(oracle_mod):
    M, K, N = 16, 48, 40
    w = si.make_workload("t", M, (K, N, N), gated=True)
    X, (Wg, Wu, W2) = si.draw(w, seed=6)
    x, wg, wu = (f32(si.bits(t)) for t in (X, Wg, Wu))
    # gate and up swapped, or the gate's SiLU dropped: both must fall outside the bound
    _, Hs = oracle_mod.chain(si.bits(X), [si.bits(Wu), si.bits(Wg), si.bits(W2)], gated=True,
                             return_h=True)
    assert not gated_bound_ok(Hs, x, wg, wu)[0]
    prod = (exact_matmul(x, wg) * exact_matmul(x, wu)).astype(np.float32)
    assert not gated_bound_ok(oracle_mod.round_bf16(prod), x, wg, wu)[0]


def test_gated_chain_zero_gate_is_exactly_zero(oracle_mod):
    # SiLU(0) = 0: a zero gate matrix zeroes H, and with it Y, bit for bit
    X, (Wg, Wu, W2) = si.draw_integer(8, (64, 32, 16), seed=7, gated=True)
    Y, H = oracle_mod.chain(si.bits(X), [np.zeros_like(si.bits(Wg)), si.bits(Wu), si.bits(W2)], gated=True,
                            return_h=True)
    assert not np.any(f32(H)) and not np.any(f32(Y))


# ------------------------------------------------------------------------------ the chain ----
def exact_matmul(a, b):
    """float64 matrix of exactly-summed (math.fsum) products; inputs are bf16 values as floats."""
    M, K = a.shape
    N = b.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            out[i, j] = math.fsum(float(a[i, k]) * float(b[k, j]) for k in range(K))
    return out


def stage_bound_ok(got_bits, a, b):
    """|got - exact| <= 2^-8 (|exact| + g A) + g A, g = K u / (1 - K u), A = sum |a b| (fp32 error bound
    for any order of K additions, plus half a bf16 ulp of rounding)."""
    K = a.shape[1]
    u = 2.0 ** -24
    g = K * u / (1 - K * u)
    exact = exact_matmul(a, b)
    A = np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64))
    got = f32(got_bits).astype(np.float64)
    bound = 2.0 ** -8 * (np.abs(exact) + g * A) + g * A
    return bool(np.all(np.abs(got - exact) <= bound)), float(np.max(np.abs(got - exact) - bound))


@pytest.mark.parametrize("M,K,N1,N2", [(16, 32, 24, 40), (9, 64, 64, 16), (32, 48, 40, 56)])
def test_chain_vs_exact_triple_loop(oracle_mod, M, K, N1, N2):
    w = si.make_workload("t", M, (K, N1, N2), x_std=1.0)
    X, (W1, W2) = si.draw(w, seed=3)
    Y, H = oracle_mod.chain(si.bits(X), [si.bits(W1), si.bits(W2)], return_h=True, threads=2)
    x, w1, w2 = f32(si.bits(X)), f32(si.bits(W1)), f32(si.bits(W2))
    ok, excess = stage_bound_ok(H, x, w1)
    assert ok, excess
    ok, excess = stage_bound_ok(Y, f32(H), w2)
    assert ok, excess


def test_chain_planted_mistakes_fail_the_pin(oracle_mod):
    M, K, N = 16, 40, 40
    w = si.make_workload("t", M, (K, N, N), x_std=1.0)
    X, (W1, W2) = si.draw(w, seed=5)
    x, w1 = f32(si.bits(X)), f32(si.bits(W1))
    # transposed operand
    Ht = oracle_mod.chain(si.bits(X), [si.bits(W1).T.copy()], threads=1)
    assert not stage_bound_ok(Ht, x, w1)[0]
    # dropped term: zero the last column of X and the last row of W1 changes nothing; zero one term
    xd = si.bits(X).copy()
    xd[:, 0] = 0
    Hd = oracle_mod.chain(xd, [si.bits(W1)], threads=1)
    assert not stage_bound_ok(Hd, x, w1)[0]
    # flipped sign of one operand row
    w1s = si.bits(W1).copy()
    w1s[3, :] ^= 0x8000
    Hs = oracle_mod.chain(si.bits(X), [w1s], threads=1)
    assert not stage_bound_ok(Hs, x, w1)[0]


@pytest.mark.parametrize("M,d", [(48, 256), (7, 1024)])
def test_chain_integer_valued_is_exact(oracle_mod, M, d):
    X, (W1, W2) = si.draw_integer(M, (d, d, d), seed=11)
    Y, H = oracle_mod.chain(si.bits(X), [si.bits(W1), si.bits(W2)], return_h=True, threads=3)
    xi = X.to(torch.int64).numpy()
    h_int = xi @ W1.to(torch.int64).numpy()
    h_bf = torch.from_numpy(h_int.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(H, si.bits(h_bf))
    y_int = h_bf.to(torch.int64).numpy() @ W2.to(torch.int64).numpy()
    assert np.abs(y_int).max() < 2 ** 24
    assert np.array_equal(Y, si.bits(torch.from_numpy(y_int.astype(np.float32)).to(torch.bfloat16)))


def test_chain_identity_and_permutation_closed_forms(oracle_mod):
    M, d = 24, 128
    X, _ = si.draw(si.make_workload("t", M, (d, d, d)), seed=7)
    I = torch.eye(d, dtype=torch.bfloat16)
    Y = oracle_mod.chain(si.bits(X), [si.bits(I), si.bits(I)])
    assert np.array_equal(Y, si.bits(X))
    P, perm = si.permutation_matrix(d, seed=2)
    Y = oracle_mod.chain(si.bits(X), [si.bits(I), si.bits(P)])
    expect = torch.empty_like(X)
    expect[:, perm] = X
    assert np.array_equal(Y, si.bits(expect))
    # power-of-two scalings are exact: (X * 2I) * (P / 2) = X P
    Y = oracle_mod.chain(si.bits(X), [si.bits((2 * I.float()).to(torch.bfloat16)),
                                      si.bits(si.permutation_matrix(d, seed=2, scale=0.5)[0])])
    assert np.array_equal(Y, si.bits(expect))
    # the transposed permutation must not pass
    Yt = oracle_mod.chain(si.bits(X), [si.bits(I), si.bits(P.T.contiguous())])
    assert not np.array_equal(Yt, si.bits(expect))


def test_chain_gelu_residual_closed_forms(oracle_mod):
    M, d = 12, 64
    X, _ = si.draw(si.make_workload("t", M, (d, d, d)), seed=9)
    Z = torch.zeros(d, d, dtype=torch.bfloat16)
    I = torch.eye(d, dtype=torch.bfloat16)
    # zero weights: gelu(0) = 0 in every stage, so the residual leaves exactly X
    Y = oracle_mod.chain(si.bits(X), [si.bits(Z)] * 4, gelu=True, residual=True)
    assert np.array_equal(Y, si.bits(X))
    # identity weights, no residual: one stage is bf16(gelu(x)); compare with torch in float64
    Y = oracle_mod.chain(si.bits(X), [si.bits(I)], gelu=True)
    ref = torch.nn.functional.gelu(X.double(), approximate="tanh")
    diff = np.abs(f32(Y).astype(np.float64) - ref.numpy())
    assert np.all(diff <= 2.0 ** -8 * np.abs(ref.numpy()) + 1e-30)
    # identity weights with residual: bf16(gelu(x) + x)
    Y = oracle_mod.chain(si.bits(X), [si.bits(I)], gelu=True, residual=True)
    ref = ref + X.double()
    diff = np.abs(f32(Y).astype(np.float64) - ref.numpy())
    assert np.all(diff <= 2.0 ** -8 * np.abs(ref.numpy()) + 2.0 ** -20)


def test_chain_row_subset_equals_full(oracle_mod):
    w = si.make_workload("t", 37, (64, 96, 32))
    X, Ws = si.draw(w, seed=4)
    full = oracle_mod.chain(si.bits(X), [si.bits(t) for t in Ws], threads=4)
    rows = np.array([0, 5, 17, 36], dtype=np.int64)
    part = oracle_mod.chain(si.bits(X), [si.bits(t) for t in Ws], rows=rows, threads=2)
    assert np.array_equal(part, full[rows])


# -------------------------------------------------------------------------- dependencies ----
def read_golden_deps(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=", 1)
                vals[k.strip()] = [int(t) for t in v.split()]
    return vals


def test_deps_tiny_golden(oracle_mod):
    g = read_golden_deps(os.path.join(GOLDEN, "deps_tiny_m64_d256_t64.txt"))
    off, tgt, init = oracle_mod.deps(64, 256, 256, 64, 64, 64, 64)
    assert off.tolist() == g["prod_off"]
    assert tgt.tolist() == g["prod_tgt"]
    assert init.tolist() == g["init_count"]


SHAPES = [
    # M, Nout, Nnext, BMp, BNp, BMc, BNc
    (64, 256, 256, 64, 64, 64, 64),
    (128, 512, 256, 128, 64, 128, 128),
    (300, 192, 160, 128, 64, 128, 32),
    (300, 200, 100, 64, 48, 128, 64),     # ragged everywhere, different row tiles
    (257, 96, 64, 128, 32, 64, 64),
    (1, 64, 64, 128, 64, 128, 64),
    (513, 128, 384, 128, 128, 128, 256),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_deps_closed_form_and_invariants(oracle_mod, shape):
    M, No, Nn, BMp, BNp, BMc, BNc = shape
    off, tgt, init = oracle_mod.deps(*shape)
    Pm, Pn = -(-M // BMp), -(-No // BNp)
    Cm, Cn = -(-M // BMc), -(-Nn // BNc)
    assert off.shape[0] == Pm * Pn + 1 and init.shape[0] == Cm * Cn
    assert off[-1] == tgt.shape[0] == init.sum()
    for c in range(Cm * Cn):
        mc = c // Cn
        r0, r1 = mc * BMc, min(M, (mc + 1) * BMc)
        row_tiles = (r1 - 1) // BMp - r0 // BMp + 1       # producer row tiles the rows touch
        assert init[c] == row_tiles * Pn
    for p in range(Pm * Pn):
        lst = tgt[off[p]:off[p + 1]].tolist()
        assert lst == sorted(set(lst))
        mp = p // Pn
        pr0, pr1 = mp * BMp, min(M, (mp + 1) * BMp)
        expect = [c for c in range(Cm * Cn)
                  if max(pr0, (c // Cn) * BMc) < min(pr1, min(M, (c // Cn + 1) * BMc))]
        assert lst == expect
