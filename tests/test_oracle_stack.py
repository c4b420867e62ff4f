"""Pins of the float64 block-stack reference (oracle/stack.py), no GPU."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc
from oracle import stack as ost


def _r(seed):
    return torch.Generator().manual_seed(seed)


def test_rowpar_pcr_matches_c_oracle():
    g = _r(1)
    for t, N, K, h, s in [(2, 5, 8, 7, 3), (4, 3, 16, 12, 0), (3, 4, 9, 6, 6), (8, 2, 64, 24, 12)]:
        X = torch.randn(N, K, generator=g, dtype=torch.float64)
        W = torch.randn(K, h, generator=g, dtype=torch.float64)
        got = ost.rowpar_pcr(X, W, t, s).numpy()
        want, _ = orc.rowpar_fwd(X.numpy(), W.numpy(), t, np.arange(s))
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_attention_matches_library_sdpa():
    g = _r(2)
    q, k, v = (torch.randn(2, 3, 7, 8, generator=g, dtype=torch.float64) for _ in range(3))
    want = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    torch.testing.assert_close(ost.causal_attention(q, k, v), want, rtol=1e-12, atol=1e-12)


def test_layer_norm_and_gelu_match_library():
    g = _r(3)
    x = torch.randn(5, 16, generator=g, dtype=torch.float64)
    w = torch.randn(16, generator=g, dtype=torch.float64)
    b = torch.randn(16, generator=g, dtype=torch.float64)
    torch.testing.assert_close(ost.layer_norm(x, w, b), F.layer_norm(x, (16,), w, b), rtol=1e-12, atol=1e-12)
    torch.testing.assert_close(ost.gelu(x), F.gelu(x), rtol=1e-12, atol=1e-12)


def test_rope_properties():
    g = _r(4)
    S, hd = 9, 8
    q = torch.randn(S, hd, generator=g, dtype=torch.float64)
    k = torch.randn(S, hd, generator=g, dtype=torch.float64)
    rq, rk = ost.rope(q), ost.rope(k)
    torch.testing.assert_close(rq[0], q[0])                    # position 0: identity
    torch.testing.assert_close(rq.norm(dim=-1), q.norm(dim=-1))  # rotations keep norms
    # rotary property: <rope(x)_m, rope(y)_n> depends on m - n only
    x = torch.randn(hd, generator=g, dtype=torch.float64)
    y = torch.randn(hd, generator=g, dtype=torch.float64)
    X = ost.rope(x.expand(S, hd).clone())
    Y = ost.rope(y.expand(S, hd).clone())
    d1 = float(X[5] @ Y[3])
    d2 = float(X[7] @ Y[5])
    assert abs(d1 - d2) < 1e-12


def _tiny_params(t=2, h=8, heads=2, ffn=16, vocab=16, layers=1, seed=5):
    g = _r(seed)
    p = {"emb": torch.randn(vocab, h, generator=g, dtype=torch.float64) * 0.5,
         "ln_f.weight": 1 + 0.1 * torch.randn(h, generator=g, dtype=torch.float64),
         "ln_f.bias": 0.1 * torch.randn(h, generator=g, dtype=torch.float64)}
    for i in range(layers):
        pre = "blocks.%d." % i
        p[pre + "ln1.weight"] = 1 + 0.1 * torch.randn(h, generator=g, dtype=torch.float64)
        p[pre + "ln1.bias"] = 0.1 * torch.randn(h, generator=g, dtype=torch.float64)
        p[pre + "ln2.weight"] = 1 + 0.1 * torch.randn(h, generator=g, dtype=torch.float64)
        p[pre + "ln2.bias"] = 0.1 * torch.randn(h, generator=g, dtype=torch.float64)
        p[pre + "wqkv"] = 0.3 * torch.randn(h, 3 * h, generator=g, dtype=torch.float64)
        p[pre + "w1"] = 0.3 * torch.randn(h, ffn, generator=g, dtype=torch.float64)
        p[pre + "wo"] = 0.3 * torch.randn(h, h, generator=g, dtype=torch.float64)
        p[pre + "w2"] = 0.3 * torch.randn(h, ffn, generator=g, dtype=torch.float64)
    return p


def test_full_reduce_keeps_ranks_identical_and_empty_set_does_not():
    t, h, heads = 2, 8, 2
    P = {k.split(".", 2)[2]: v for k, v in _tiny_params().items() if k.startswith("blocks.0.")}
    g = _r(6)
    x = torch.randn(3, h, generator=g, dtype=torch.float64)
    x = torch.stack([x, x])                       # identical streams going in
    y1 = ost.block(x, P, t, heads, h, 1, 3)        # S = all channels: vanilla transformer
    torch.testing.assert_close(y1[0], y1[1], rtol=0, atol=0)
    y0 = ost.block(x, P, t, heads, 0, 1, 3)        # S empty: the ranks drift apart
    assert (y0[0] - y0[1]).abs().max() > 1e-3


def test_loss_gradients_match_finite_differences():
    t, heads, layers = 2, 2, 1
    params = _tiny_params()
    tokens = torch.tensor([[1, 5, 3, 9], [2, 2, 7, 0]])
    L, grads = ost.loss_and_grads(params, tokens, t, heads, layers, 4)
    eps = 1e-6
    for name, idx in [("blocks.0.wo", (1, 2)), ("blocks.0.w2", (3, 5)), ("blocks.0.wqkv", (1, 20)),
                      ("emb", (5, 1)), ("blocks.0.ln1.weight", (3,))]:
        pp = {k: v.clone() for k, v in params.items()}
        pm = {k: v.clone() for k, v in params.items()}
        pp[name][idx] += eps
        pm[name][idx] -= eps
        fd = (float(ost.loss(pp, tokens, t, heads, layers, 4)) - float(ost.loss(pm, tokens, t, heads, layers, 4))) / (2 * eps)
        assert abs(fd - float(grads[name][idx])) <= 1e-6 * (1 + abs(fd)), name


SHARDED = ("wqkv", "wo", "w1", "w2")


def test_column_placement_at_empty_set_is_the_exact_gradient():
    # S empty: neither placement reduces anything, so the column placement's
    # explicit backward must equal autograd's exact gradient.
    t, heads, layers = 2, 2, 2
    params = _tiny_params(layers=layers)
    tokens = torch.tensor([[1, 5, 3, 9], [2, 2, 7, 0]])
    L0, g0 = ost.loss_and_grads(params, tokens, t, heads, layers, 0)
    L1, g1 = ost.loss_and_grads(params, tokens, t, heads, layers, 0, "column")
    assert L0 == L1
    for k in params:
        torch.testing.assert_close(g1[k], g0[k], rtol=1e-10, atol=1e-12)


def test_column_placement_at_full_set_is_megatron():
    # S full: every rank carries the same stream, the model is the vanilla
    # transformer, and the exact gradient is its gradient.  Megatron's placement
    # back-propagates 1/t of the loss gradient on each rank (the loss averages the
    # t identical streams) and reduces only at the column-parallel inputs: the
    # replicated parameters, summed over ranks, get the exact gradient, and each
    # sharded weight, used by one rank only, gets exactly 1/t of it.
    t, heads, layers = 2, 2, 2
    params = _tiny_params(layers=layers)
    tokens = torch.tensor([[1, 5, 3, 9], [2, 2, 7, 0]])
    h = params["emb"].shape[1]
    _, g0 = ost.loss_and_grads(params, tokens, t, heads, layers, h)
    _, g1 = ost.loss_and_grads(params, tokens, t, heads, layers, h, "column")
    for k in params:
        scale = 1.0 / t if k.split(".")[-1] in SHARDED else 1.0
        torch.testing.assert_close(g1[k], scale * g0[k], rtol=1e-9, atol=1e-12)


def test_column_placement_differs_at_partial_set():
    # 0 < p < 1 with a norm between the layers: the placements differ (they are
    # different readings, not one gradient computed two ways)
    t, heads, layers = 2, 2, 1
    params = _tiny_params(layers=layers)
    tokens = torch.tensor([[1, 5, 3, 9], [2, 2, 7, 0]])
    _, g0 = ost.loss_and_grads(params, tokens, t, heads, layers, 4)
    _, g1 = ost.loss_and_grads(params, tokens, t, heads, layers, 4, "column")
    assert (g1["blocks.0.w1"] - g0["blocks.0.w1"]).abs().max() > 1e-6


def test_column_layer_matches_c_oracle():
    g = _r(11)
    for t, N, h, K, s in [(2, 5, 6, 8, 3), (4, 3, 8, 16, 0), (3, 4, 6, 9, 6)]:
        A = torch.randn(t, N, h, generator=g, dtype=torch.float64, requires_grad=True)
        W1 = torch.randn(h, K, generator=g, dtype=torch.float64, requires_grad=True)
        dZ = torch.randn(N, K, generator=g, dtype=torch.float64)
        Z = ost.ColReduce.apply(A, W1, t, s)
        Z.backward(dZ)
        np.testing.assert_allclose(Z.detach().numpy(), orc.colpar_fwd(A.detach().numpy(), W1.detach().numpy(), t),
                                   rtol=1e-12, atol=1e-12)
        wA, wW = orc.colpar_bwd(A.detach().numpy(), W1.detach().numpy(), dZ.numpy(), t, np.arange(s))
        np.testing.assert_allclose(A.grad.numpy(), wA, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(W1.grad.numpy(), wW, rtol=1e-12, atol=1e-12)


def test_rowpar_pcr_index_list_matches_c_oracle():
    # S as a list of channels (a seeded random subset): the same sums as the C oracle
    g = _r(11)
    rng = np.random.default_rng(12)
    for t, N, K, h, s in [(2, 5, 8, 7, 3), (4, 3, 16, 12, 5), (8, 2, 64, 24, 12)]:
        S = np.sort(rng.permutation(h)[:s]).astype(np.int32)
        X = torch.randn(N, K, generator=g, dtype=torch.float64)
        W = torch.randn(K, h, generator=g, dtype=torch.float64)
        got = ost.rowpar_pcr(X, W, t, S).numpy()
        want, _ = orc.rowpar_fwd(X.numpy(), W.numpy(), t, S)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
        # channels outside S keep the rank's own partial: they differ between ranks
        out = np.setdiff1d(np.arange(h), S)
        assert np.abs(got[0][:, out] - got[1][:, out]).max() > 1e-6


def _relabel(params, perm):
    """The stack's parameters with the residual-stream channels renamed: new channel
    j is old channel perm[j].  Every h-indexed axis moves: the embedding's columns,
    the norms' gains and biases, and the rows of the four weights (QKV and MLP-up
    read the stream, out- and down-projection write it)."""
    out = {}
    for k, v in params.items():
        leaf = k.split(".")[-1]
        if k == "emb":
            out[k] = v[:, perm]
        elif leaf in ("weight", "bias"):
            out[k] = v[perm]
        else:
            out[k] = v[perm, :]
    return out


@pytest.mark.parametrize("placement", ["reduce_dout", "column"])
def test_random_set_equals_contiguous_set_after_relabelling(placement):
    # Every op of the block either acts channel-wise on the stream (norm gains,
    # residual adds, the partial reduce) or sums over all its channels (norm
    # statistics, the QKV / MLP-up contractions), so renaming the channels -- S
    # first -- leaves the loss unchanged and renames the gradients the same way.
    t, heads, layers, h = 2, 2, 2, 8
    params = _tiny_params(layers=layers)
    tokens = torch.tensor([[1, 5, 3, 9], [2, 2, 7, 0]])
    S = np.array([1, 4, 6], dtype=np.int32)
    perm = np.concatenate([S, np.setdiff1d(np.arange(h), S)])
    L_r, g_r = ost.loss_and_grads(params, tokens, t, heads, layers, S, placement)
    L_c, g_c = ost.loss_and_grads(_relabel(params, perm), tokens, t, heads, layers, len(S), placement)
    assert abs(L_r - L_c) <= 1e-12 * abs(L_r)
    g_rp = _relabel(g_r, perm)
    for k in params:
        torch.testing.assert_close(g_c[k], g_rp[k], rtol=1e-9, atol=1e-12)
    # and the random set is not the contiguous one: the loss differs without the renaming
    L_x, _ = ost.loss_and_grads(params, tokens, t, heads, layers, len(S), placement)
    assert abs(L_x - L_r) > 1e-9
