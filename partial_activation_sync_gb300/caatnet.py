"""CAAT-Net block stack on one GPU, the t tensor-parallel ranks emulated in one HBM.

"Tensor-Parallelism with Partially Synchronized Activations" (NeurIPS 2025),
Introduction: every tensor-parallel all-reduce of the transformer -- after the
attention out-projection and after the MLP down-projection, Megatron's two
row-parallel layers per block -- becomes a partial channel-reduce, so the
activations of the ranks differ and the residual stream is kept as t copies
[t, N, h].  Experiments: the 130M model has h = 768, 16 heads, 12 layers,
sequence 1024; p = 0.5, tensor-parallel dimension 8.

Readings where the pages are silent:
  * GPT-style pre-norm blocks: LayerNorm, causal multi-head attention with rotary
    position embeddings, a GELU MLP of width FFN (3072 = 4h), tied input/output
    embeddings;
  * column-parallel layers (QKV, MLP up) give rank r its heads / its FFN slice,
    computed from rank r's own residual copy;
  * the row-parallel layers run the library's fused GEMM + partial reduce.  Where
    the backward reduce sits is a reading ("forward and backward must agree"):
    placement "reduce_dout" (default) is the exact gradient, the row-parallel
    backward reducing its upstream gradient over S; placement "column" is
    Megatron's, the row-parallel backward passing each rank's gradient through and
    the column-parallel layers (QKV, MLP up) reducing their input gradient over S
    in the library's column-parallel backward;
  * norm weights and the embedding are replicated: one parameter used by all ranks;
  * the loss needs one full reduction ("communicating only to compute the loss"):
    the ranks' final residual copies are averaged, then LayerNorm, the tied LM head
    and next-token cross-entropy.

The row-parallel and column-parallel layers run in this library's kernels;
attention, norms, GELU, embedding and loss are PyTorch ops of the harness.  Column-parallel weights are stored [h, K] with column
block r owned by rank r (K contiguous: the layout the library's kernels take).

S is the first round(p h) channels by default, or a seeded random subset
(layout="random"), which the layers receive as an index list.  A random S costs
the layers a pass over their outputs (the forward) and over the upstream gradient
(the backward) that a contiguous S does not.  relabel_channels() removes that
cost: it renames the residual stream's channels so that S comes first, which
gives a model with a contiguous S that computes the same loss.
"""

import numpy as np
import torch
import torch.nn as nn
import torch.nn.functional as F

from . import (CAAT_BWD_NO_REDUCE, CAAT_BWD_REDUCE_DOUT, CAAT_S_CONTIGUOUS, CAAT_S_RANDOM,
               colpar_linear_bwd, colpar_linear_fwd, rowpar_linear_bwd, rowpar_linear_fwd,
               select_channels)


class RowParallelPCR(torch.autograd.Function):
    """Y[r] = PCR_S(X_r W_r) for the t ranks (rank r's input is column block r of X).

    X: [N, K]; W: logical [K, h] (an nn.Linear weight [h, K] passed as .t());
    sel: S as a device index tensor or an int n (S = first n channels);
    mode: the backward's CAAT_BWD_REDUCE_DOUT or CAAT_BWD_NO_REDUCE.
    Returns Y [t, N, h]."""

    @staticmethod
    def forward(ctx, X, W, t, sel, mode=CAAT_BWD_REDUCE_DOUT):
        N = X.shape[0]
        h = W.shape[1]
        Y = torch.empty((t, N, h), dtype=X.dtype, device=X.device)
        rowpar_linear_fwd(X, W, t, sel, outs=list(Y.unbind(0)))
        ctx.save_for_backward(X, W)
        ctx.t, ctx.sel, ctx.mode = t, sel, mode
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, W = ctx.saved_tensors
        dY = dY.contiguous()
        dX, dW = rowpar_linear_bwd(X, W, list(dY.unbind(0)), ctx.t, ctx.sel, ctx.mode)
        return dX, dW, None, None, None


class ColParallelPCR(torch.autograd.Function):
    """Z[:, block r] = A_r W1_r for the t ranks (A [t, N, h]: rank r's own input;
    W1 [h, K], block r of its columns = rank r's).  The backward reduces the input
    gradient over S: dA_r = PCR_S(dZ_r W1_r^T).  Returns Z [N, K]."""

    @staticmethod
    def forward(ctx, A, W1, t, sel):
        ctx.save_for_backward(A, W1)
        ctx.t, ctx.sel = t, sel
        return colpar_linear_fwd(A, W1, t)

    @staticmethod
    def backward(ctx, dZ):
        A, W1 = ctx.saved_tensors
        dA, dW1 = colpar_linear_bwd(A, W1, dZ.contiguous(), ctx.t, ctx.sel)
        return dA, dW1, None, None


def rope_tables(seq, hd, device, dtype, base=10000.0):
    inv = 1.0 / (base ** (torch.arange(0, hd, 2, device=device, dtype=torch.float32) / hd))
    ang = torch.arange(seq, device=device, dtype=torch.float32)[:, None] * inv[None, :]
    return ang.cos().to(dtype), ang.sin().to(dtype)


def apply_rope(x, cos, sin):
    """x [..., S, hd]: rotate the pairs (x[2i], x[2i+1]) by the angle of position and i."""
    x1, x2 = x[..., 0::2], x[..., 1::2]
    r1 = x1 * cos - x2 * sin
    r2 = x1 * sin + x2 * cos
    return torch.stack((r1, r2), dim=-1).flatten(-2)


PLACEMENTS = ("reduce_dout", "column")


class Block(nn.Module):
    def __init__(self, h, heads, ffn, t, std=0.02, placement="reduce_dout"):
        super().__init__()
        assert heads % t == 0 and ffn % t == 0 and h % heads == 0 and placement in PLACEMENTS
        self.h, self.heads, self.ffn, self.t = h, heads, ffn, t
        self.placement = placement
        self.hd = h // heads
        self.ln1 = nn.LayerNorm(h)
        self.ln2 = nn.LayerNorm(h)
        # column-parallel, [in = h, out = K]; column block r = rank r's heads / FFN slice
        self.wqkv = nn.Parameter(torch.randn(h, 3 * h) * std)
        self.w1 = nn.Parameter(torch.randn(h, ffn) * std)
        # row-parallel, nn.Linear layout [out = h, in = K]; K shard r = rank r's heads / FFN slice
        self.wo = nn.Parameter(torch.randn(h, h) * std)
        self.w2 = nn.Parameter(torch.randn(h, ffn) * std)

    def _colpar(self, a, W1, sel):
        """[t, N, h] -> [t, N, K/t]: rank r's input times its column block, in the
        library's column-parallel kernels.  Placement "column" reduces the input
        gradient over S; the default placement reduces nothing there (an empty S:
        each rank's input gradient is its own dZ_r W1_r^T)."""
        t, N, h = a.shape
        kt = W1.shape[1] // t
        sel = sel if self.placement == "column" else 0
        return ColParallelPCR.apply(a, W1, t, sel).view(N, t, kt).transpose(0, 1)

    def forward(self, x, cos, sin, batch, seq, sel):
        """x [t, N, h]: the ranks' residual streams; sel: S (a channel count or a
        device index tensor)."""
        t, N, h = x.shape
        hpr = self.heads // t                              # heads per rank
        mode = CAAT_BWD_NO_REDUCE if self.placement == "column" else CAAT_BWD_REDUCE_DOUT
        qkv = self._colpar(self.ln1(x), self.wqkv, sel)    # [t, N, 3 h/t]
        qkv = qkv.reshape(t, batch, seq, 3, hpr, self.hd).permute(3, 0, 1, 4, 2, 5)
        q, k, v = (z.reshape(t * batch, hpr, seq, self.hd) for z in qkv)
        q, k = apply_rope(q, cos, sin), apply_rope(k, cos, sin)
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)   # [t*B, hpr, S, hd]
        o = o.view(t, batch, hpr, seq, self.hd).permute(1, 3, 0, 2, 4).reshape(N, h)
        x = x + RowParallelPCR.apply(o, self.wo.t(), t, sel, mode)
        u = F.gelu(self._colpar(self.ln2(x), self.w1, sel))   # [t, N, ffn/t]
        u = u.transpose(0, 1).reshape(N, self.ffn)         # column block r = rank r
        return x + RowParallelPCR.apply(u, self.w2.t(), t, sel, mode)


class CAATNet(nn.Module):
    """Token ids [batch, seq] -> mean next-token cross-entropy.

    layout "contiguous": S = the first round(p h) channels, passed to the layers by
    its size; "random": a seeded random subset of that size, passed as an index
    list (kept as an int32 buffer that moves with the model)."""

    def __init__(self, vocab=32000, h=768, heads=16, layers=12, ffn=3072, t=8, p=0.5, seq=1024,
                 std=0.02, placement="reduce_dout", layout="contiguous", seed=0):
        super().__init__()
        assert layout in ("contiguous", "random")
        self.t, self.h, self.heads, self.seq = t, h, heads, seq
        self.placement = placement
        kind = CAAT_S_RANDOM if layout == "random" else CAAT_S_CONTIGUOUS
        self.S = select_channels(h, p, kind, seed)         # sorted channel indices of S
        self.n_sel = int(self.S.size)
        # an index list only where it says more than a count: 0 < |S| < h and not
        # the first |S| channels
        contiguous = bool(np.array_equal(self.S, np.arange(self.n_sel)))
        self.register_buffer("sel_idx", None if contiguous else torch.from_numpy(self.S.copy()),
                             persistent=False)
        self.emb = nn.Parameter(torch.randn(vocab, h) * std)
        self.blocks = nn.ModuleList([Block(h, heads, ffn, t, std, placement) for _ in range(layers)])
        self.ln_f = nn.LayerNorm(h)

    def sel(self):
        """S as the layers take it: the index buffer, or the count of a contiguous S."""
        return self.sel_idx if self.sel_idx is not None else self.n_sel

    def forward(self, tokens):
        batch, seq = tokens.shape
        N = batch * seq
        x0 = F.embedding(tokens.reshape(N), self.emb)      # [N, h], identical on every rank
        x = x0.unsqueeze(0).expand(self.t, N, self.h).contiguous()
        cos, sin = rope_tables(seq, self.h // self.heads, x.device, x.dtype)
        sel = self.sel()
        for blk in self.blocks:
            x = blk(x, cos, sin, batch, seq, sel)
        z = self.ln_f(x.mean(dim=0))                       # the reduction the loss needs
        logits = z @ self.emb.t()                          # tied LM head
        tgt = tokens.reshape(batch, seq)[:, 1:].reshape(-1)
        logits = logits.view(batch, seq, -1)[:, :-1].reshape(-1, logits.shape[-1])
        return F.cross_entropy(logits.float(), tgt)


def channel_order(S, h):
    """The renaming that puts S first: new channel j is old channel perm[j] (S in
    ascending order, then the other channels in ascending order)."""
    S = np.asarray(S, dtype=np.int64)
    return np.concatenate([S, np.setdiff1d(np.arange(h), S)])


@torch.no_grad()
def relabel_channels(model):
    """A model with a contiguous S (the first |S| channels) that computes the same
    loss as ``model`` with its S, and its gradients renamed.

    Every op of a block acts on the residual stream either channel by channel (the
    norms' gains and biases, the residual adds, the partial reduce) or by summing
    over all its channels (the norms' statistics, the QKV and MLP-up
    contractions), so renaming the channels commutes with the model.  What moves is
    every axis indexed by a stream channel: the embedding's columns (also the tied
    LM head), the norms' gains and biases, and the rows of the four weights (QKV
    and MLP-up read the stream, out- and down-projection write it).  Only the
    order of floating-point sums over channels changes.  Returns (new model, perm)
    with new channel j = old channel perm[j]."""
    blk0 = model.blocks[0]
    new = CAATNet(vocab=model.emb.shape[0], h=model.h, heads=model.heads, layers=len(model.blocks),
                  ffn=blk0.ffn, t=model.t, p=model.n_sel / model.h, seq=model.seq,
                  placement=model.placement, layout="contiguous")
    assert new.n_sel == model.n_sel
    new = new.to(device=model.emb.device, dtype=model.emb.dtype)
    perm = channel_order(model.S, model.h)
    ix = torch.from_numpy(perm).to(model.emb.device)
    src = dict(model.named_parameters())
    for name, p in new.named_parameters():
        q = src[name]
        leaf = name.split(".")[-1]
        if name == "emb":
            p.copy_(q[:, ix])
        elif leaf in ("weight", "bias"):
            p.copy_(q[ix])
        else:
            p.copy_(q[ix, :])
    return new, perm


def train_step(model, opt, tokens):
    """One training step: forward, backward, AdamW update.  Returns the loss (device)."""
    opt.zero_grad(set_to_none=True)
    loss = model(tokens)
    loss.backward()
    opt.step()
    return loss.detach()
