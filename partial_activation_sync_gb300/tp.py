"""Tensor parallelism across processes (one GPU each) with the partial
channel-reduce as the only exchange.

"Tensor-Parallelism with Partially Synchronized Activations" (NeurIPS 2025),
Introduction: after a row-parallel layer the all-reduce of the activations is
replaced by the partial channel-reduce, which sums only the channels of S over
the tensor-parallel ranks; the other channels stay with their rank.  The
reproducibility card's inference setup runs this over NVLink GPUs.  Here the
t ranks of the layer may be spread over P processes (one GPU each), t/P ranks
per GPU:

  1. each process runs the fused forward of its own t/P shards, which already
     sums its local ranks' partials on S (one GPU, no exchange);
  2. the channels of S of that local sum go through a rank-ordered all-reduce
     across the processes: a dense [N, |S|] buffer is cut into P blocks of rows,
     an all-to-all hands block q of every process to process q, which folds the
     P blocks in process order (fp32, one rounding: the result does not depend on
     the split), and an all-gather returns every folded block to everyone;
  3. the reduced channels are written back into every local rank's output.
  The channels outside S never leave their GPU.  Bytes sent per process:
  2 (P-1)/P N |S| elem, the p-fraction of what an all-reduce of all h channels
  moves (the pages' "up to 50% less communication" at p = 0.5).

With a contiguous S the exchange of step 2 overlaps the forward of the channels
outside S: the S channels are computed first into the dense buffer, and the
rest is computed on the launching stream while the exchange runs on a second one.

The steps on each GPU (pack, fold, unpack, the local forward, reduce and
backward) are the library's kernels (``LibraryOps``); only the collectives are
torch.distributed calls.  Another ``ops`` object with the same methods can
stand in for them, which is how the protocol is tested on CPU processes over
gloo.
"""
import torch
import torch.distributed as dist

from . import (CAAT_BWD_NO_REDUCE, partial_channel_reduce, pcr_pack, pcr_unpack, rank_fold,
               rowpar_linear_bwd, rowpar_linear_fwd)


class LibraryOps:
    """The per-GPU steps as this library's CUDA kernels."""

    @staticmethod
    def pack(Y, sel, P):
        pcr_pack(Y, sel, P)

    @staticmethod
    def fold(R, out):
        rank_fold(R, out)

    @staticmethod
    def unpack(P, sel, Ys):
        pcr_unpack(P, sel, Ys)

    @staticmethod
    def forward(X, W, t, sel, outs):
        rowpar_linear_fwd(X, W, t, sel, outs=outs)

    @staticmethod
    def local_reduce(dOut, sel, dY):
        partial_channel_reduce(dOut, sel, outs=dY)

    @staticmethod
    def backward(X, W, dY, t, sel, dX, dW):
        return rowpar_linear_bwd(X, W, dY, t, sel, CAAT_BWD_NO_REDUCE, dX=dX, dW=dW)


def _n_sel(sel):
    return int(sel) if isinstance(sel, int) else int(sel.numel())


def _bytes(x):
    """A contiguous tensor seen as bytes (collectives move bits, not values)."""
    return x.reshape(-1).view(torch.uint8)


class PartialReduce:
    """Rank-ordered sum of the channels of S across the processes of `group`.

    Buffers are kept per shape and reused; the padding rows of the send buffer
    (when the token count is not a multiple of the process count) stay zero."""

    def __init__(self, group=None, ops=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.ops = ops if ops is not None else LibraryOps()
        self.nccl = dist.get_backend(group) == "nccl"
        self._bufs = {}

    def send_buffer(self, N, s, dtype, device):
        """The dense [P * C, s] buffer (C = ceil(N / P)) whose first N rows the
        caller fills with this process's S channels."""
        return self._buf("P", N, s, dtype, device)

    def _buf(self, name, N, s, dtype, device):
        C = -(-N // self.world)
        key = (name, N, s, dtype, str(device))
        b = self._bufs.get(key)
        if b is None:
            shape = {"P": (self.world * C, s), "R": (self.world, C, s), "red": (C, s),
                     "G": (self.world * C, s)}[name]
            b = torch.zeros(shape, dtype=dtype, device=device)
            self._bufs[key] = b
        return b

    def exchange(self, P, N):
        """All-reduce (rank-ordered fold) of the send buffer P; returns the reduced
        [P * C, s] buffer whose first N rows are the result."""
        if self.world == 1:
            return P
        s = P.shape[1]
        R = self._buf("R", N, s, P.dtype, P.device)
        red = self._buf("red", N, s, P.dtype, P.device)
        G = self._buf("G", N, s, P.dtype, P.device)
        # block q of every process's rows goes to process q
        dist.all_to_all_single(_bytes(R), _bytes(P), group=self.group)
        self.ops.fold(R, red)
        if self.nccl:
            dist.all_gather_into_tensor(_bytes(G), _bytes(red), group=self.group)
        else:
            dist.all_gather(list(_bytes(G).chunk(self.world)), _bytes(red), group=self.group)
        return G

    def __call__(self, Ys, sel):
        """Sum the channels of S of this process's outputs Ys (a list of [N, h]
        tensors that agree on S) over the processes; writes the sum into the S
        channels of every tensor of Ys."""
        N = Ys[0].shape[0]
        s = _n_sel(sel)
        if s == 0 or N == 0:
            return Ys
        P = self.send_buffer(N, s, Ys[0].dtype, Ys[0].device)
        self.ops.pack(Ys[0], sel, P[:N])
        G = self.exchange(P, N)
        self.ops.unpack(G[:N], sel, Ys)
        return Ys


def rowpar_linear_fwd_tp(X, W, t_local, sel, pr, outs=None, side=None):
    """Row-parallel layer + partial channel-reduce with the t ranks spread over
    the processes of ``pr`` (a PartialReduce), t_local ranks on this GPU.

    X: [N, t_local * k_t], this process's shards of the input (rank order);
    W: logical [t_local * k_t, h], the matching rows of the weight (e.g.
    ``linear.weight[:, cols].t()``).  sel: the channels of S (int s for the
    first s channels, else an int32 index tensor), the same on every process.
    Returns the t_local outputs [N, h]: channels of S hold the sum over all t
    ranks of every process, the other channels each local rank's own partial.
    side: the stream for the exchange (contiguous S only; default: a new one)."""
    N = X.shape[0]
    h = W.shape[1]
    if outs is None:
        outs = [torch.empty((N, h), dtype=X.dtype, device=X.device) for _ in range(t_local)]
    s = _n_sel(sel)
    ops = pr.ops
    if not isinstance(sel, int) or s == 0 or s == h or pr.world == 1:
        ops.forward(X, W, t_local, sel, outs)
        if pr.world > 1:
            pr(outs, sel)
        return outs
    # contiguous S: the S channels first, summed over the local shards (one
    # output: a single rank over all local K), into the dense send buffer
    P = pr.send_buffer(N, s, X.dtype, X.device)
    ops.forward(X, W[:, :s], 1, s, [P[:N]])
    if not X.is_cuda:
        G = pr.exchange(P, N)
        ops.unpack(G[:N], s, outs)
        ops.forward(X, W[:, s:], t_local, 0, [y[:, s:] for y in outs])
        return outs
    main = torch.cuda.current_stream()
    side = side if side is not None else torch.cuda.Stream(device=X.device)
    side.wait_stream(main)
    with torch.cuda.stream(side):
        G = pr.exchange(P, N)
        ops.unpack(G[:N], s, outs)
    # meanwhile the channels outside S, each local rank its own partial
    ops.forward(X, W[:, s:], t_local, 0, [y[:, s:] for y in outs])
    main.wait_stream(side)
    return outs


def rowpar_linear_bwd_tp(X, W, dOut, t_local, sel, pr, dX=None, dW=None, dY=None):
    """Backward of ``rowpar_linear_fwd_tp`` with the reduce on the upstream
    gradient (the exact gradient of sum_r <dOut_r, Y_r>): dY = PCR(dOut) over all
    t ranks, then this process's dX [N, t_local k_t] and dW (W's layout).

    The local ranks' gradients are reduced on S by the library's partial reduce
    into dY (t_local buffers [N, h], allocated when None), that local sum goes
    through the exchange across processes, and the GEMMs then run on dY in the
    no-reduce placement.  Returns (dX, dW)."""
    N, h = dOut[0].shape
    if dY is None:
        dY = [torch.empty((N, h), dtype=dOut[0].dtype, device=dOut[0].device) for _ in range(t_local)]
    pr.ops.local_reduce(dOut, sel, dY)
    if pr.world > 1:
        pr(dY, sel)
    return pr.ops.backward(X, W, dY, t_local, sel, dX, dW)
