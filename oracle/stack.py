"""Float64 CPU reference of the CAAT-Net block stack -- TEST INFRASTRUCTURE ONLY.

Written independently of the product package (which it never imports): plain
PyTorch CPU ops in float64, autograd for the gradients.

"Tensor-Parallelism with Partially Synchronized Activations" (NeurIPS 2025),
Introduction: each tensor-parallel all-reduce of the transformer (after the
attention out-projection and the MLP down-projection) is replaced by the partial
channel-reduce, so the t ranks carry different residual streams.  The readings of
the unstated architecture (pre-norm GPT block with LayerNorm, rotary attention,
GELU MLP, tied embeddings; ranks' final streams averaged for the loss) are the same
ones the product documents.  The column-parallel weights (QKV, MLP up) are
[h, K] with column block r owned by rank r.

Two placements of the backward reduce ("forward and backward must agree" does not
say where it sits):
  * "reduce_dout": the exact gradient of the forward (plain autograd): the
    row-parallel backward reduces its upstream gradient over S;
  * "column": Megatron's placement: the row-parallel backward passes each rank's
    gradient through unreduced and the column-parallel layer reduces its input
    gradient over S.  Written out with explicit backward formulas below; it is not
    the gradient of the forward when 0 < p < 1.
"""
import math

import numpy as np
import torch


def in_s(h, s, dtype):
    """Membership of the h channels in S as 0/1 of the given dtype.  S is a subset
    of the channels (Introduction, partial channel-reduce): an int s stands for the
    first s channels, an integer array for the listed channels."""
    if isinstance(s, (int, np.integer)):
        return (torch.arange(h) < int(s)).to(dtype)
    m = torch.zeros(h, dtype=dtype)
    m[torch.as_tensor(np.asarray(s, dtype=np.int64))] = 1
    return m


def rowpar_pcr(X, W, t, s):
    """X [N, K], W [K, h]; rank r's partial sum X_r W_r over shard r of K; the
    channels of S (see in_s) summed over ranks in rank order, the rest rank-local.
    Returns [t, N, h]."""
    K = X.shape[1]
    kt = K // t
    parts = [X[:, r * kt:(r + 1) * kt] @ W[r * kt:(r + 1) * kt] for r in range(t)]
    total = parts[0]
    for r in range(1, t):
        total = total + parts[r]
    inS = in_s(W.shape[1], s, X.dtype)
    return torch.stack([inS * total + (1 - inS) * parts[r] for r in range(t)])


def _blocks(K, t):
    kt = K // t
    return [slice(r * kt, (r + 1) * kt) for r in range(t)]


class RowNoReduce(torch.autograd.Function):
    """rowpar_pcr in the forward; the backward back-propagates each rank's own
    gradient through X_r W_r (no reduce: it moves to the column-parallel layer)."""

    @staticmethod
    def forward(ctx, X, W, t, s):
        ctx.save_for_backward(X, W)
        ctx.t = t
        return rowpar_pcr(X, W, t, s)

    @staticmethod
    def backward(ctx, G):
        X, W = ctx.saved_tensors
        bl = _blocks(X.shape[1], ctx.t)
        dX = torch.cat([G[r] @ W[b].t() for r, b in enumerate(bl)], dim=1)
        dW = torch.cat([X[:, b].t() @ G[r] for r, b in enumerate(bl)], dim=0)
        return dX, dW, None, None


class ColReduce(torch.autograd.Function):
    """Column-parallel layer: A [t, N, h] (rank r's own input), W1 [h, K];
    Z[:, block r] = A_r W1[:, block r].  Backward: the input gradient of rank r is
    P_r = dZ_r W1_r^T, reduced over the channels of S (left fold in rank order,
    the sum given to every rank); the rest stay each rank's own."""

    @staticmethod
    def forward(ctx, A, W1, t, s):
        ctx.save_for_backward(A, W1)
        ctx.t, ctx.s = t, s
        return torch.cat([A[r] @ W1[:, b] for r, b in enumerate(_blocks(W1.shape[1], t))], dim=1)

    @staticmethod
    def backward(ctx, dZ):
        A, W1 = ctx.saved_tensors
        t, s = ctx.t, ctx.s
        bl = _blocks(W1.shape[1], t)
        P = [dZ[:, b] @ W1[:, b].t() for b in bl]
        total = P[0]
        for r in range(1, t):
            total = total + P[r]
        inS = in_s(W1.shape[0], s, A.dtype)
        dA = torch.stack([inS * total + (1 - inS) * P[r] for r in range(t)])
        dW1 = torch.cat([A[r].t() @ dZ[:, b] for r, b in enumerate(bl)], dim=1)
        return dA, dW1, None, None


def layer_norm(x, g, b, eps=1e-5):
    mu = x.mean(dim=-1, keepdim=True)
    var = ((x - mu) ** 2).mean(dim=-1, keepdim=True)
    return (x - mu) / torch.sqrt(var + eps) * g + b


def gelu(x):
    return 0.5 * x * (1.0 + torch.erf(x / math.sqrt(2.0)))


def rope(x, base=10000.0):
    """x [..., S, hd]: pair (2i, 2i+1) at position m rotated by m * base^(-2i/hd)."""
    S, hd = x.shape[-2], x.shape[-1]
    i = torch.arange(hd // 2, dtype=torch.float64)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * base ** (-2.0 * i / hd)[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x1 * s + x2 * c
    return out


def causal_attention(q, k, v):
    """q, k, v [..., S, hd]: softmax(q k^T / sqrt(hd) with j > i masked) v."""
    S, hd = q.shape[-2], q.shape[-1]
    sc = q @ k.transpose(-1, -2) / math.sqrt(hd)
    mask = torch.triu(torch.ones(S, S, dtype=torch.bool), diagonal=1)
    sc = sc.masked_fill(mask, float("-inf"))
    return torch.softmax(sc, dim=-1) @ v


def block(x, P, t, heads, s, batch, seq, placement="reduce_dout"):
    """x [t, N, h]; P: dict of float64 parameter tensors of one block."""
    _, N, h = x.shape
    hd = h // heads
    hpr = heads // t
    a = torch.stack([layer_norm(x[r], P["ln1.weight"], P["ln1.bias"]) for r in range(t)])
    if placement == "column":
        qkv_all = ColReduce.apply(a, P["wqkv"], t, s)           # [N, 3h], block r = rank r
        row = RowNoReduce.apply
    else:
        qkv_all = torch.cat([a[r] @ P["wqkv"][:, b] for r, b in enumerate(_blocks(3 * h, t))], dim=1)
        row = rowpar_pcr
    outs = []
    for r, b in enumerate(_blocks(3 * h, t)):
        qkv = qkv_all[:, b]                                     # [N, 3 h/t]
        q, k, v = qkv.reshape(batch, seq, 3, hpr, hd).permute(2, 0, 3, 1, 4)   # [B, hpr, S, hd] each
        o = causal_attention(rope(q), rope(k), v)               # [B, hpr, S, hd]
        outs.append(o.permute(0, 2, 1, 3).reshape(N, h // t))
    o_cat = torch.cat(outs, dim=1)                              # column block r = rank r
    x = x + row(o_cat, P["wo"].t(), t, s)
    b2 = torch.stack([layer_norm(x[r], P["ln2.weight"], P["ln2.bias"]) for r in range(t)])
    ffn = P["w1"].shape[1]
    if placement == "column":
        up = ColReduce.apply(b2, P["w1"], t, s)
    else:
        up = torch.cat([b2[r] @ P["w1"][:, b] for r, b in enumerate(_blocks(ffn, t))], dim=1)
    return x + row(gelu(up), P["w2"].t(), t, s)


def loss(params, tokens, t, heads, layers, s, placement="reduce_dout"):
    """params: dict name -> float64 tensor (names as in the product's module);
    tokens [batch, seq] int64.  Mean next-token cross-entropy."""
    batch, seq = tokens.shape
    N = batch * seq
    emb = params["emb"]
    x0 = emb[tokens.reshape(N)]
    x = torch.stack([x0] * t)
    for i in range(layers):
        P = {k.split(".", 2)[2]: v for k, v in params.items() if k.startswith("blocks.%d." % i)}
        x = block(x, P, t, heads, s, batch, seq, placement)
    z = layer_norm(x.mean(dim=0), params["ln_f.weight"], params["ln_f.bias"])
    logits = (z @ emb.t()).view(batch, seq, -1)[:, :-1].reshape(-1, emb.shape[0])
    tgt = tokens[:, 1:].reshape(-1)
    logp = logits - torch.logsumexp(logits, dim=-1, keepdim=True)
    return -logp[torch.arange(tgt.numel()), tgt].mean()


def loss_and_grads(params64, tokens, t, heads, layers, s, placement="reduce_dout"):
    ps = {k: v.detach().clone().requires_grad_(True) for k, v in params64.items()}
    L = loss(ps, tokens, t, heads, layers, s, placement)
    L.backward()
    return float(L.detach()), {k: v.grad for k, v in ps.items()}
