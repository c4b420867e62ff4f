"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Definition followed: "Tensor-Parallelism with Partially Synchronized Activations"
(NeurIPS 2025), Introduction, the partial channel-reduce paragraph: a subset S
of hidden channels is summed over the t tensor-parallel ranks, the rest stay as
each rank computed them; S empty = ensemble, S full = vanilla all-reduce; the
parameter count and the compute do not change; forward and backward must agree.
The abstract and the experimental setup give the payload cut: 50% at p = 0.5.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import oracle as orc
import caat_inputs as ci

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------ golden values

def test_splitmix64_published_outputs():
    g = _load("splitmix64.json")
    for case in g["cases"]:
        want = [int(v, 0) for v in case["outputs"]]
        got = orc.splitmix64(case["seed"], len(want))
        assert [int(x) for x in got] == want


def test_bf16_rounding_hand_values():
    g = _load("bf16_rne.json")
    f = np.array([c["f32"] for c in g["cases"]], dtype=np.float32)
    want = np.array([int(c["bf16"], 16) for c in g["cases"]], dtype=np.uint16)
    np.testing.assert_array_equal(orc.f32_to_bf16(f), want)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    a = _rng(7).standard_normal(20000).astype(np.float32) * np.float32(37.0)
    # include exact halfway points between neighbouring bf16 values
    base = (_rng(8).integers(0, 2**15, 4000).astype(np.uint32) << 16) | 0x8000
    a = np.concatenate([a, base.view(np.float32)])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(orc.f32_to_bf16(a), ref)


@pytest.mark.parametrize("case", _load("pcr_hand.json")["cases"], ids=lambda c: c["name"])
def test_pcr_hand_examples(case):
    Y = np.array(case["Y"], dtype=np.float32)
    want = np.array(case["Out"], dtype=np.float32)
    out, red = orc.pcr_f32(Y, case["sel"])
    np.testing.assert_array_equal(out, want)
    assert red == case["reduced"]
    out64, red64 = orc.pcr_f64(Y.astype(np.float64), case["sel"])
    if case["name"] != "t3_fp32_left_fold_order":   # double keeps the 1
        np.testing.assert_array_equal(out64, want.astype(np.float64))
    assert red64 == case["reduced"]


def test_rowpar_hand_example():
    g = _load("rowpar_hand.json")
    X = np.array(g["X"], dtype=np.float64)
    W = np.array(g["W"], dtype=np.float64)
    t = g["t"]
    for f in g["fwd"]:
        out, _ = orc.rowpar_fwd(X, W, t, f["sel"])
        np.testing.assert_array_equal(out, np.array(f["Out"], dtype=np.float64))
    for b in g["bwd"]:
        dX, dW = orc.rowpar_bwd(X, W, np.array(b["G"], dtype=np.float64), t, b["sel"], b["mode"])
        np.testing.assert_array_equal(dX, np.array(b["dX"], dtype=np.float64))
        np.testing.assert_array_equal(dW, np.array(b["dW"], dtype=np.float64))


# ------------------------------------------------------- channel selection

@pytest.mark.parametrize("h", range(0, 13))
def test_select_channels_brute_force(h):
    for layout in (0, 1):
        for seed in (0, 1, 12345):
            prev = None
            for k in range(h + 1):
                p = k / h if h else 0.0
                S = orc.select_channels(h, p, layout, seed)
                assert S.size == k
                assert np.all(np.diff(S) > 0)
                assert S.size == 0 or (S.min() >= 0 and S.max() < h)
                if layout == 0:
                    np.testing.assert_array_equal(S, np.arange(k))
                if prev is not None:   # nesting: S(p1) is a subset of S(p2) for p1 < p2
                    assert set(prev.tolist()) <= set(S.tolist())
                prev = S


def test_select_channels_rounding_half_up():
    # s = floor(p*h + 1/2)
    assert orc.select_channels(10, 0.25, 0).size == 3     # 2.5 -> 3
    assert orc.select_channels(10, 0.24, 0).size == 2     # 2.4 -> 2
    assert orc.select_channels(768, 0.5, 0).size == 384
    assert orc.select_channels(4096, 0.75, 1, 4003).size == 3072
    with pytest.raises(ValueError):
        orc.select_channels(8, 1.5, 0)
    with pytest.raises(ValueError):
        orc.select_channels(8, 0.5, 2)


def test_select_channels_random_is_a_uniform_shuffle():
    # With h = 3 the nested sets S(1/3), S(2/3) reveal the first two shuffle
    # entries, hence the whole permutation.  A correct Fisher-Yates makes all 3! = 6
    # permutations equally likely; the classic slip j = rand mod h (instead of
    # mod (i+1)) makes them 4/27, 5/27, ... and fails this chi-square test.
    counts = {}
    n = 6000
    for seed in range(n):
        a = orc.select_channels(3, 1 / 3, 1, seed)
        b = orc.select_channels(3, 2 / 3, 1, seed)
        first = int(a[0])
        second = int(sorted(set(b.tolist()) - {first})[0])
        third = ({0, 1, 2} - {first, second}).pop()
        counts[(first, second, third)] = counts.get((first, second, third), 0) + 1
    assert len(counts) == 6
    exp = n / 6
    chi2 = sum((c - exp) ** 2 / exp for c in counts.values())
    assert chi2 < 20.5   # chi-square, 5 dof, p = 0.001


def test_select_channels_random_differs_by_seed():
    a = orc.select_channels(2048, 0.5, 1, 4003)
    b = orc.select_channels(2048, 0.5, 1, 4004)
    assert a.size == b.size == 1024
    assert not np.array_equal(a, b)
    # a random half of 2048 channels is far from the contiguous block
    assert len(set(a.tolist()) & set(range(1024))) < 600


# --------------------------------------------------- partial channel-reduce

def test_pcr_integer_values_match_exact_sum():
    r = _rng(1)
    t, N, h = 5, 7, 33
    Y = r.integers(-1000, 1000, size=(t, N, h)).astype(np.float32)
    S = np.array(sorted(r.choice(h, 12, replace=False)), dtype=np.int32)
    out, red = orc.pcr_f32(Y, S)
    tot = Y.astype(np.int64).sum(axis=0)
    for rr in range(t):
        np.testing.assert_array_equal(out[rr][:, S], tot[:, S].astype(np.float32))
        notS = np.setdiff1d(np.arange(h), S)
        np.testing.assert_array_equal(out[rr][:, notS], Y[rr][:, notS])
    assert red == N * S.size


def test_pcr_f32_left_fold_bitexact_random():
    # the fold order is ours (the paper does not fix it): compare with numpy's
    # explicit sequential adds in float32
    r = _rng(2)
    t, N, h = 8, 9, 40
    Y = r.standard_normal((t, N, h)).astype(np.float32)
    S = orc.select_channels(h, 0.5, 1, 99)
    out, _ = orc.pcr_f32(Y, S)
    acc = Y[0].copy()
    for q in range(1, t):
        acc = (acc + Y[q]).astype(np.float32)
    for rr in range(t):
        np.testing.assert_array_equal(out[rr][:, S], acc[:, S])


def test_pcr_bf16_is_f32_fold_then_one_rounding():
    torch = pytest.importorskip("torch")
    r = _rng(3)
    t, N, h = 4, 6, 48
    Yf = r.standard_normal((t, N, h)).astype(np.float32)
    Yb = torch.from_numpy(Yf).to(torch.bfloat16)
    Ywords = Yb.view(torch.int16).numpy().view(np.uint16)
    S = orc.select_channels(h, 0.5, 0)
    out, red = orc.pcr_bf16(Ywords, S)
    acc = Yb[0].float()
    for q in range(1, t):
        acc = acc + Yb[q].float()
    accw = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for rr in range(t):
        np.testing.assert_array_equal(out[rr][:, S], accw[:, S])
        notS = np.setdiff1d(np.arange(h), S)
        np.testing.assert_array_equal(out[rr][:, notS], Ywords[rr][:, notS])
    assert red == N * S.size


def test_pcr_adjoint_identity():
    # PCR is symmetric: <PCR(A), B> = <A, PCR(B)>, which is what lets the same
    # operator serve as its own backward.
    r = _rng(4)
    for t, h, p in [(2, 7, 0.5), (3, 11, 0.3), (5, 16, 1.0), (4, 9, 0.0)]:
        A = r.standard_normal((t, 3, h))
        B = r.standard_normal((t, 3, h))
        S = orc.select_channels(h, p, 1, 5)
        lhs = np.sum(orc.pcr_f64(A, S)[0] * B)
        rhs = np.sum(A * orc.pcr_f64(B, S)[0])
        assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))


def test_pcr_payload_is_p_of_allreduce():
    # communicated elements: N*|S| = p * (N*h); 50% at p = 0.5
    t, N, h = 8, 16, 768
    Y = _rng(5).standard_normal((t, N, h)).astype(np.float32)
    for p in (0.0, 0.25, 0.5, 0.75, 1.0):
        S = orc.select_channels(h, p, 0)
        _, red = orc.pcr_f32(Y, S)
        assert red == round(p * N * h)


# ------------------------------------------------- row-parallel linear layer

def _shards(X, W, t):
    K = X.shape[1]
    kt = K // t
    return [(X[:, r * kt:(r + 1) * kt], W[r * kt:(r + 1) * kt]) for r in range(t)]


@pytest.mark.parametrize("t,N,K,h", [(1, 3, 4, 5), (2, 4, 6, 7), (3, 5, 9, 8), (4, 2, 16, 12)])
def test_rowpar_fwd_limits_match_numpy(t, N, K, h):
    r = _rng(10 + t)
    X = r.standard_normal((N, K))
    W = r.standard_normal((K, h))
    # p = 1: vanilla all-reduce, every rank holds X @ W
    out, macs = orc.rowpar_fwd(X, W, t, np.arange(h))
    full = X @ W
    for rr in range(t):
        np.testing.assert_allclose(out[rr], full, rtol=1e-12, atol=1e-12)
    assert macs == N * K * h
    # p = 0: ensemble, rank r holds its own partial sum X_r @ W_r
    out0, macs0 = orc.rowpar_fwd(X, W, t, [])
    for rr, (Xr, Wr) in enumerate(_shards(X, W, t)):
        np.testing.assert_allclose(out0[rr], Xr @ Wr, rtol=1e-12, atol=1e-12)
    assert macs0 == macs


def test_rowpar_fwd_mixed_set_matches_einsum():
    r = _rng(20)
    t, N, K, h = 4, 5, 12, 10
    X = r.standard_normal((N, K))
    W = r.standard_normal((K, h))
    S = orc.select_channels(h, 0.5, 1, 77)
    out, macs = orc.rowpar_fwd(X, W, t, S)
    Y = np.einsum("nrk,rkc->rnc", X.reshape(N, t, K // t), W.reshape(t, K // t, h))
    for rr in range(t):
        for c in range(h):
            want = Y[:, :, c].sum(axis=0) if c in S else Y[rr, :, c]
            np.testing.assert_allclose(out[rr, :, c], want, rtol=1e-12, atol=1e-12)
    # S columns are bit-identical on every rank
    for rr in range(1, t):
        assert np.array_equal(out[rr][:, S], out[0][:, S])
    assert macs == N * K * h   # compute unchanged by p


def test_rowpar_fwd_closed_form_ones():
    # X = 1, W = 1: a partial sum is K/t, a reduced channel is K
    t, N, K, h = 8, 3, 64, 16
    S = orc.select_channels(h, 0.5, 1, 3)
    out, _ = orc.rowpar_fwd(np.ones((N, K)), np.ones((K, h)), t, S)
    for c in range(h):
        want = K if c in S else K // t
        assert np.all(out[:, :, c] == want)


def test_parameter_count_independent_of_p():
    t, K, h = 8, 768, 768
    W = np.zeros((K, h))
    sizes = [Wr.size for _, Wr in _shards(np.zeros((1, K)), W, t)]
    assert sum(sizes) == K * h


def _loss(X, W, G, t, S):
    out, _ = orc.rowpar_fwd(X, W, t, S)
    return float(np.sum(out * G))


@pytest.mark.parametrize("t,N,K,h,p", [(2, 3, 4, 5, 0.0), (2, 4, 6, 7, 0.5), (3, 5, 6, 7, 0.5),
                                         (3, 2, 9, 4, 1.0), (2, 1, 2, 3, 0.34)])
def test_rowpar_bwd_matches_finite_differences(t, N, K, h, p):
    # The loss L = sum_r <G_r, Out_r> is bilinear in (X, W): central differences
    # are exact up to rounding, so this pins dX and dW of the reduce-dOut mode.
    r = _rng(30 + N)
    X = r.standard_normal((N, K))
    W = r.standard_normal((K, h))
    G = r.standard_normal((t, N, h))
    S = orc.select_channels(h, p, 1, 11)
    dX, dW = orc.rowpar_bwd(X, W, G, t, S, orc.REDUCE_DOUT)
    eps = 1e-3
    for idx in itertools.product(range(N), range(K)):
        Xp = X.copy(); Xp[idx] += eps
        Xm = X.copy(); Xm[idx] -= eps
        fd = (_loss(Xp, W, G, t, S) - _loss(Xm, W, G, t, S)) / (2 * eps)
        assert abs(fd - dX[idx]) <= 1e-8 * (1 + abs(fd))
    for idx in itertools.product(range(K), range(h)):
        Wp = W.copy(); Wp[idx] += eps
        Wm = W.copy(); Wm[idx] -= eps
        fd = (_loss(X, Wp, G, t, S) - _loss(X, Wm, G, t, S)) / (2 * eps)
        assert abs(fd - dW[idx]) <= 1e-8 * (1 + abs(fd))


def test_rowpar_bwd_no_reduce_is_the_local_gradient():
    # mode NO_REDUCE: each rank back-propagates its own G_r through X_r W_r --
    # the gradient of sum_r <G_r, X_r W_r>, i.e. the S-empty layer, for any S
    r = _rng(40)
    t, N, K, h = 3, 4, 9, 6
    X = r.standard_normal((N, K))
    W = r.standard_normal((K, h))
    G = r.standard_normal((t, N, h))
    S = orc.select_channels(h, 0.5, 0)
    dX, dW = orc.rowpar_bwd(X, W, G, t, S, orc.NO_REDUCE)
    dX0, dW0 = orc.rowpar_bwd(X, W, G, t, [], orc.REDUCE_DOUT)
    np.testing.assert_array_equal(dX, dX0)
    np.testing.assert_array_equal(dW, dW0)
    kt = K // t
    for rr in range(t):
        np.testing.assert_allclose(dX[:, rr * kt:(rr + 1) * kt], G[rr] @ W[rr * kt:(rr + 1) * kt].T,
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dW[rr * kt:(rr + 1) * kt], X[:, rr * kt:(rr + 1) * kt].T @ G[rr],
                                   rtol=1e-12, atol=1e-12)


def test_rowpar_bwd_full_set_is_allreduce_gradient():
    # p = 1: every rank's gradient on the reduced output is the sum of the G_r
    r = _rng(41)
    t, N, K, h = 4, 3, 8, 5
    X = r.standard_normal((N, K))
    W = r.standard_normal((K, h))
    G = r.standard_normal((t, N, h))
    dX, dW = orc.rowpar_bwd(X, W, G, t, np.arange(h), orc.REDUCE_DOUT)
    Gs = G.sum(axis=0)
    np.testing.assert_allclose(dX, Gs @ W.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dW, X.T @ Gs, rtol=1e-12, atol=1e-12)


def test_rowpar_rejects_indivisible_k():
    with pytest.raises(ValueError):
        orc.rowpar_fwd(np.ones((2, 5)), np.ones((5, 3)), 2, [0])


def test_bf16_input_widening_is_exact():
    a = ci.normal(5, (1000,))
    w = ci.bf16_words(a)
    np.testing.assert_array_equal(orc.bf16_to_f64(w), ci.words_to_f32(w).astype(np.float64))
    np.testing.assert_array_equal(orc.f32_to_bf16(ci.words_to_f32(w)), w)
