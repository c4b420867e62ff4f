"""The partial channel-reduce across processes (partial_activation_sync_gb300.tp)
over gloo on CPU processes, world sizes 2 and 3.

The protocol -- the dense send buffer with its padding rows, the all-to-all of
row blocks, the fold in process order, the all-gather, the write-back into every
local rank's output, and the split of a contiguous S from the channels outside
it -- is the product's code.  The per-process steps that run as CUDA kernels on a
GPU (pack, fold, unpack, the local fused forward) are stood in for here by the
oracle on CPU tensors; on the GPU those kernels are checked against the same
oracle functions in tests/test_gpu_exchange.py.

Expected values are computed independently in every process from the seeded
inputs: each process's local output is the oracle's row-parallel forward of its
own shards, rounded to the dtype; the channels of S must then hold, bit for bit,
the oracle's partial channel-reduce (left fold in process order) of the
processes' local S sums, and every other channel its own rank's value."""
import os
import socket

import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc

T_LOCAL_SEED = 7000


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class OracleOps:
    """Per-process steps on CPU tensors, from the oracle (stand-ins for the kernels)."""

    def __init__(self, dtype):
        self.dtype = dtype

    @staticmethod
    def _idx(sel, h):
        return np.arange(int(sel)) if isinstance(sel, int) else sel.numpy().astype(np.int64)

    def pack(self, Y, sel, P):
        P.copy_(Y[:, self._idx(sel, Y.shape[1])])

    def fold(self, R, out):
        import torch
        t, rows, cols = R.shape
        allc = np.arange(cols, dtype=np.int32)
        if R.dtype == torch.bfloat16:
            w = R.contiguous().view(torch.int16).numpy().view(np.uint16)
            o = orc.pcr_bf16(w, allc)[0][0]
            out.copy_(torch.from_numpy(o.view(np.int16).copy()).view(torch.bfloat16))
        else:
            o = orc.pcr_f32(R.contiguous().numpy(), allc)[0][0]
            out.copy_(torch.from_numpy(o.copy()))

    def unpack(self, P, sel, Ys):
        idx = self._idx(sel, Ys[0].shape[1])
        for y in Ys:
            y[:, idx] = P

    def local_reduce(self, dOut, sel, dY):
        import torch
        S = self._idx(sel, dOut[0].shape[1]).astype(np.int32)
        if dOut[0].dtype == torch.bfloat16:
            w = np.stack([d.contiguous().view(torch.int16).numpy().view(np.uint16) for d in dOut])
            o = orc.pcr_bf16(w, S)[0]
            for r in range(len(dY)):
                dY[r].copy_(torch.from_numpy(o[r].view(np.int16).copy()).view(torch.bfloat16))
        else:
            o = orc.pcr_f32(np.stack([d.numpy() for d in dOut]), S)[0]
            for r in range(len(dY)):
                dY[r].copy_(torch.from_numpy(o[r].copy()))

    def backward(self, X, W, dY, t, sel, dX, dW):
        S = self._idx(sel, W.shape[1]).astype(np.int32)
        gX, gW = orc.rowpar_bwd(X.double().numpy(), W.double().numpy(),
                                np.stack([d.double().numpy() for d in dY]), t, S, 1)
        return _round(gX, X.dtype), _round(gW, X.dtype)

    def forward(self, X, W, t, sel, outs):
        import torch
        h = W.shape[1]
        S = self._idx(sel, h).astype(np.int32)
        out, _ = orc.rowpar_fwd(X.double().numpy(), W.double().numpy(), t, S)
        for r in range(t):
            outs[r].copy_(_round(out[r], X.dtype))


def _round(a64, dtype):
    """float64 -> the tensor dtype (through float32, then bf16 nearest-even)."""
    import torch
    f = np.asarray(a64, dtype=np.float32)
    if dtype == torch.bfloat16:
        return torch.from_numpy(orc.f32_to_bf16(f).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(f)


def _inputs(world, t_local, N, kt, h, dtype):
    """Full seeded X [N, K] and W [K, h] (K = world * t_local * kt) as the dtype's values."""
    K = world * t_local * kt
    X = ci.normal(T_LOCAL_SEED + 1, (N, K))
    W = ci.normal(T_LOCAL_SEED + 2, (K, h), std=0.02)
    if dtype == "bf16":
        X = ci.words_to_f32(ci.bf16_words(X))
        W = ci.words_to_f32(ci.bf16_words(W))
    return X.astype(np.float64), W.astype(np.float64)


def _worker(rank, world, port, case, q):
    try:
        import torch
        import torch.distributed as dist
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from partial_activation_sync_gb300 import tp
        t_local, N, kt, h, p, layout, dname = case
        tdt = torch.bfloat16 if dname == "bf16" else torch.float32
        X, W = _inputs(world, t_local, N, kt, h, dname)
        S = orc.select_channels(h, p, layout, 4321)
        sel = int(S.size) if layout == 0 else torch.from_numpy(S)
        kl = t_local * kt
        cols = slice(rank * kl, (rank + 1) * kl)
        Xl = _round(X[:, cols], tdt)
        Wl = _round(W[cols, :], tdt)
        pr = tp.PartialReduce(ops=OracleOps(dname))
        outs = tp.rowpar_linear_fwd_tp(Xl, Wl, t_local, sel, pr)
        got = [o.float().numpy().astype(np.float64) for o in outs]

        # expected, from the oracle alone: every process's local sum on S ...
        def local(g):
            c = slice(g * kl, (g + 1) * kl)
            o, _ = orc.rowpar_fwd(X[:, c], W[c, :], t_local, S)
            return o
        locs = [local(g) for g in range(world)]
        mine = locs[rank]
        if dname == "bf16":
            words = np.stack([orc.f32_to_bf16(np.asarray(l_[0], dtype=np.float32)) for l_ in locs])
            red = orc.pcr_bf16(words, S)[0][0]
            red = orc.bf16_to_f64(red)
            own = [orc.bf16_to_f64(orc.f32_to_bf16(np.asarray(mine[r], dtype=np.float32))) for r in range(t_local)]
        else:
            vals = np.stack([np.asarray(l_[0], dtype=np.float32) for l_ in locs])
            red = orc.pcr_f32(vals, S)[0][0].astype(np.float64)
            own = [np.asarray(mine[r], dtype=np.float32).astype(np.float64) for r in range(t_local)]
        notS = np.setdiff1d(np.arange(h), S)
        ok = True
        for r in range(t_local):
            ok &= np.array_equal(got[r][:, S], red[:, S])          # bit for bit
            ok &= np.array_equal(got[r][:, notS], own[r][:, notS])
        # ... and within the bf16 / fp32 tolerance of the plain definition
        full, _ = orc.rowpar_fwd(X, W, world * t_local, S)
        rel = max(float(np.linalg.norm(got[r] - full[rank * t_local + r]) / np.linalg.norm(full[rank * t_local + r]))
                  for r in range(t_local))
        # the backward (reduce on the upstream gradient) against the plain definition
        t = world * t_local
        Gf = ci.normal(T_LOCAL_SEED + 3, (t, N, h))
        if dname == "bf16":
            Gf = ci.words_to_f32(ci.bf16_words(Gf))
        Gf = Gf.astype(np.float64)
        dOut = [_round(Gf[rank * t_local + r], tdt) for r in range(t_local)]
        gX, gW = tp.rowpar_linear_bwd_tp(Xl, Wl, dOut, t_local, sel, pr)
        wX, wW = orc.rowpar_bwd(X, W, Gf, t, S, 0)
        gXv, gWv = gX.double().numpy(), gW.double().numpy()
        rel_b = max(float(np.linalg.norm(gXv - wX[:, cols]) / np.linalg.norm(wX[:, cols])),
                    float(np.linalg.norm(gWv - wW[cols, :]) / np.linalg.norm(wW[cols, :])))
        q.put((rank, bool(ok), max(rel, rel_b)))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        import traceback
        q.put((rank, False, "%s\n%s" % (e, traceback.format_exc())))


CASES = [
    # world, t_local, N, k_t, h, p, layout, dtype
    (2, 2, 37, 16, 40, 0.5, 0, "bf16"),    # contiguous S: S first, exchange, then the rest
    (2, 2, 37, 16, 40, 0.5, 1, "bf16"),    # random S: local forward, pack, exchange, unpack
    (3, 1, 20, 8, 24, 0.5, 0, "f32"),      # one rank per process; 20 rows over 3 processes
    (3, 2, 29, 8, 24, 0.25, 1, "bf16"),
    (2, 1, 16, 8, 24, 1.0, 0, "bf16"),     # S = every channel: the all-reduce
    (2, 2, 16, 8, 24, 0.0, 0, "bf16"),     # S empty: no exchange at all
]


@pytest.mark.parametrize("case", CASES)
def test_partial_reduce_across_processes_gloo(case):
    import torch.multiprocessing as mp
    world = case[0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case[1:], q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
    tol = 1e-2 if case[-1] == "bf16" else 1e-5
    for rank, ok, rel in res:
        assert ok is True, (rank, rel)
        assert rel <= tol, (rank, rel)
    assert all(pr.exitcode == 0 for pr in procs)


def _bytes_worker(rank, world, port, N, h, ps, q):
    """Count the bytes this process hands to the collectives for one exchange per p."""
    try:
        import torch
        import torch.distributed as dist
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from partial_activation_sync_gb300 import tp
        sent = {"n": 0}
        a2a, ag = dist.all_to_all_single, dist.all_gather

        def count_a2a(out, inp, *a, **k):
            # every block but this process's own leaves it
            sent["n"] += inp.numel() * inp.element_size() * (world - 1) // world
            return a2a(out, inp, *a, **k)

        def count_ag(outs, inp, *a, **k):
            # this process's block goes to every other process
            sent["n"] += inp.numel() * inp.element_size() * (world - 1)
            return ag(outs, inp, *a, **k)

        dist.all_to_all_single, dist.all_gather = count_a2a, count_ag
        res = []
        for p in ps:
            S = orc.select_channels(h, p, 0, 0)
            Y = [torch.from_numpy(ci.normal(9000 + rank, (N, h))).to(torch.bfloat16)]
            sent["n"] = 0
            tp.PartialReduce(ops=OracleOps("bf16"))(Y, int(S.size))
            res.append(sent["n"])
        dist.all_to_all_single, dist.all_gather = a2a, ag
        q.put((rank, res))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover
        import traceback
        q.put((rank, "%s\n%s" % (e, traceback.format_exc())))


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_bytes_are_the_p_fraction_of_an_all_reduce(world):
    """The pages' communication claim ("up to 50% less" at p = 0.5): each process
    sends 2 (P-1)/P N |S| elem bytes, where a ring all-reduce of all h channels
    sends 2 (P-1)/P N h elem -- the ratio is p exactly (N a multiple of P)."""
    import torch.multiprocessing as mp
    N, h, ps = 64, 96, (0.25, 0.5, 1.0)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bytes_worker, args=(r, world, port, N, h, ps, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
    allreduce = 2 * (world - 1) * N * h * 2 // world
    for rank, counts in res:
        assert isinstance(counts, list), counts
        for p, n in zip(ps, counts):
            s = int(p * h + 0.5)
            assert n == 2 * (world - 1) * N * s * 2 // world, (rank, p, n)
            assert n / allreduce == pytest.approx(p), (rank, p)
