"""Pins of the CPU oracle's column-parallel layer (no GPU needed).

"Tensor-Parallelism with Partially Synchronized Activations" (NeurIPS 2025),
Introduction: the partial channel-reduce replaces the tensor-parallel all-reduce,
and forward and backward must agree.  In Megatron's placement the backward reduce
sits on the input gradient of the column-parallel layer (QKV, MLP up).  Reading
used here: the input channels in S are one activation shared by the ranks and the
others are each rank's own, so the exact gradient with respect to those logical
variables is the reduce over S of the ranks' input gradients.  The finite
differences below pin exactly that; p = 0 and p = 1 reduce to library matmuls.
"""
import itertools

import numpy as np
import pytest

from oracle import oracle as orc


def _rng(seed):
    return np.random.default_rng(seed)


def _blocks(K, t):
    kt = K // t
    return [slice(r * kt, (r + 1) * kt) for r in range(t)]


@pytest.mark.parametrize("t,N,h,K", [(1, 3, 4, 5), (2, 4, 5, 6), (4, 3, 7, 8), (3, 5, 2, 9)])
def test_colpar_fwd_matches_numpy(t, N, h, K):
    r = _rng(100 + t)
    A = r.standard_normal((t, N, h))
    W1 = r.standard_normal((h, K))
    Z = orc.colpar_fwd(A, W1, t)
    for rr, b in enumerate(_blocks(K, t)):
        np.testing.assert_allclose(Z[:, b], A[rr] @ W1[:, b], rtol=1e-12, atol=1e-12)


def test_colpar_bwd_limits_match_numpy():
    r = _rng(101)
    t, N, h, K = 4, 5, 6, 8
    A = r.standard_normal((t, N, h))
    W1 = r.standard_normal((h, K))
    dZ = r.standard_normal((N, K))
    bl = _blocks(K, t)
    # p = 0: each rank's input gradient is its own dZ_r W1_r^T
    dA, dW1 = orc.colpar_bwd(A, W1, dZ, t, [])
    for rr, b in enumerate(bl):
        np.testing.assert_allclose(dA[rr], dZ[:, b] @ W1[:, b].T, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dW1[:, b], A[rr].T @ dZ[:, b], rtol=1e-12, atol=1e-12)
    # p = 1: the all-reduce gives every rank the unsharded layer's gradient dZ W1^T
    dA1, dW11 = orc.colpar_bwd(A, W1, dZ, t, np.arange(h))
    for rr in range(t):
        np.testing.assert_allclose(dA1[rr], dZ @ W1.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(dW1, dW11)     # dW1 does not depend on S


def test_colpar_bwd_s_channels_identical_across_ranks():
    r = _rng(102)
    t, N, h, K = 3, 4, 10, 9
    A = r.standard_normal((t, N, h))
    W1 = r.standard_normal((h, K))
    dZ = r.standard_normal((N, K))
    S = orc.select_channels(h, 0.5, 1, 7)
    dA, _ = orc.colpar_bwd(A, W1, dZ, t, S)
    for rr in range(1, t):
        np.testing.assert_array_equal(dA[rr][:, S], dA[0][:, S])
    notS = np.setdiff1d(np.arange(h), S)
    assert not np.array_equal(dA[1][:, notS], dA[0][:, notS])


def _assemble(shared, priv, S, t, N, h):
    """Per-rank inputs from the logical variables: S channels shared, the rest own."""
    notS = np.setdiff1d(np.arange(h), S)
    A = np.empty((t, N, h))
    for rr in range(t):
        A[rr][:, S] = shared
        A[rr][:, notS] = priv[rr]
    return A, notS


def colpar_logical_fd_errors(bwd, t, N, h, K, p, seed):
    """Largest |finite difference - analytic| over every logical input and W1
    entry, for the loss L = <G, Z>; bwd(A, W1, G, t, S) -> (dA, dW1)."""
    r = _rng(seed)
    S = orc.select_channels(h, p, 1, seed)
    shared = r.standard_normal((N, S.size))
    priv = r.standard_normal((t, N, h - S.size))
    W1 = r.standard_normal((h, K))
    G = r.standard_normal((N, K))
    A, notS = _assemble(shared, priv, S, t, N, h)
    dA, dW1 = bwd(A, W1, G, t, S)

    def loss(sh, pv, w):
        a, _ = _assemble(sh, pv, S, t, N, h)
        return float(np.sum(orc.colpar_fwd(a, w, t) * G))

    eps = 1e-3
    err = 0.0
    for idx in itertools.product(range(N), range(S.size)):
        p_, m_ = shared.copy(), shared.copy()
        p_[idx] += eps
        m_[idx] -= eps
        fd = (loss(p_, priv, W1) - loss(m_, priv, W1)) / (2 * eps)
        for rr in range(t):
            err = max(err, abs(fd - dA[rr][idx[0], S[idx[1]]]) / (1 + abs(fd)))
    for idx in itertools.product(range(t), range(N), range(h - S.size)):
        p_, m_ = priv.copy(), priv.copy()
        p_[idx] += eps
        m_[idx] -= eps
        fd = (loss(shared, p_, W1) - loss(shared, m_, W1)) / (2 * eps)
        err = max(err, abs(fd - dA[idx[0]][idx[1], notS[idx[2]]]) / (1 + abs(fd)))
    for idx in itertools.product(range(h), range(K)):
        p_, m_ = W1.copy(), W1.copy()
        p_[idx] += eps
        m_[idx] -= eps
        fd = (loss(shared, priv, p_) - loss(shared, priv, m_)) / (2 * eps)
        err = max(err, abs(fd - dW1[idx]) / (1 + abs(fd)))
    return err


@pytest.mark.parametrize("t,N,h,K,p", [(2, 3, 4, 4, 0.5), (3, 2, 5, 6, 0.4), (2, 2, 3, 4, 0.0),
                                         (4, 2, 3, 8, 1.0), (3, 3, 6, 3, 0.5)])
def test_colpar_bwd_matches_logical_finite_differences(t, N, h, K, p):
    # L is bilinear in (logical inputs, W1): central differences are exact up to
    # rounding, so dA on S (every rank), dA outside S and dW1 are all pinned.
    err = colpar_logical_fd_errors(orc.colpar_bwd, t, N, h, K, p, seed=110 + 7 * t + N)
    assert err <= 1e-8


def test_colpar_rejects_indivisible_k():
    with pytest.raises(ValueError):
        orc.colpar_fwd(np.ones((2, 3, 4)), np.ones((4, 5)), 2)
    with pytest.raises(ValueError):
        orc.colpar_bwd(np.ones((2, 3, 4)), np.ones((4, 5)), np.ones((3, 5)), 2, [0])
