"""The tensor-parallel split of partial_activation_sync_gb300.tp with the
library's CUDA kernels (LibraryOps), P ranks of a process group emulated as P
threads of this process on this one GPU.

The collectives are a stand-in: the threads meet at a barrier, each publishes its
send buffer once its stream has finished writing it, and each copies what the
real collective would deliver (the all-to-all's row blocks, the all-gather's
folded blocks) with device-to-device copies.  No kernel waits on another: every
exchange is host-ordered.  What runs on the GPU is exactly the product path --
the local fused forward, pack, the rank-ordered fold, unpack, and for a
contiguous S the forward of the channels outside S on the launching stream while
the exchange runs on a second one.  Results are checked against the oracle as in
tests/test_tp_host.py: bit for bit on S against the partial reduce of the
processes' local sums (each process's local forward, run on its own by the same
library calls, gives those sums and every rank's channels outside S), within
tolerance against the plain definition."""
import threading

import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import torch

pytestmark = pytest.mark.gpu


class FakeGroup:
    """P threads as the ranks of a process group (barrier-ordered copies)."""

    def __init__(self, world):
        self.world = world
        self.bar = threading.Barrier(world)
        self.slots = [None] * world
        self.local = threading.local()

    # the subset of torch.distributed that tp.py uses
    def get_world_size(self, group=None):
        return self.world

    def get_rank(self, group=None):
        return self.local.rank

    def get_backend(self, group=None):
        return "fake"

    def _publish(self, t):
        T = torch()
        T.cuda.current_stream().synchronize()        # the buffer is written
        self.slots[self.local.rank] = t
        self.bar.wait()

    def all_to_all_single(self, out, inp, group=None):
        T = torch()
        self._publish(inp)
        r, P = self.local.rank, self.world
        n = inp.numel() // P
        for q in range(P):
            out[q * n:(q + 1) * n].copy_(self.slots[q][r * n:(r + 1) * n])
        T.cuda.current_stream().synchronize()
        self.bar.wait()                                # everyone has read every slot

    def all_gather(self, outs, inp, group=None):
        T = torch()
        self._publish(inp)
        for q in range(self.world):
            outs[q].copy_(self.slots[q])
        T.cuda.current_stream().synchronize()
        self.bar.wait()


def _round_bf16(a):
    return ci.words_to_f32(ci.bf16_words(a)).astype(np.float64)


@pytest.mark.parametrize("P,t_local,N,kt,h,p,layout", [
    (2, 4, 300, 64, 512, 0.5, 0),      # contiguous S: S first, exchange on a side stream
    (4, 2, 257, 128, 256, 0.5, 1),     # random S: local forward, pack, exchange, unpack
    (8, 1, 1024, 512, 1024, 0.5, 0),   # one rank per GPU-thread (the tp8 layout)
])
def test_tp_split_on_threads_matches_oracle(P, t_local, N, kt, h, p, layout, monkeypatch):
    T = torch()
    import partial_activation_sync_gb300 as caat
    from partial_activation_sync_gb300 import tp
    fake = FakeGroup(P)
    monkeypatch.setattr(tp, "dist", fake)
    t = P * t_local
    K = t * kt
    X = ci.normal(7501, (N, K))
    W = ci.normal(7502, (K, h), std=0.02)
    S = orc.select_channels(h, p, layout, 17)
    kl = t_local * kt
    results = [None] * P
    errors = []

    def rank_main(g):
        try:
            fake.local.rank = g
            T.cuda.set_device(0)
            with T.cuda.stream(T.cuda.Stream()):
                cols = slice(g * kl, (g + 1) * kl)
                Xg = T.from_numpy(ci.bf16_words(np.ascontiguousarray(X[:, cols])).view(np.int16)).cuda().view(T.bfloat16)
                Wg = T.from_numpy(ci.bf16_words(np.ascontiguousarray(W[cols, :].T)).view(np.int16)).cuda().view(T.bfloat16)
                sel = int(S.size) if layout == 0 else T.from_numpy(S).cuda()
                # this process alone: its local sum on S and its ranks' own channels
                s = int(S.size)
                if layout == 0:
                    loc_s = caat.rowpar_linear_fwd(Xg, Wg.t()[:, :s], 1, s)[0]
                    loc = caat.rowpar_linear_fwd(Xg, Wg.t()[:, s:], t_local, 0)
                    own = [o.view(T.int16).cpu().numpy().view(np.uint16) for o in loc]
                else:
                    loc = caat.rowpar_linear_fwd(Xg, Wg.t(), t_local, sel)
                    loc_s = loc[0][:, S.tolist()]
                    own = [o.view(T.int16).cpu().numpy().view(np.uint16)[:, np.setdiff1d(np.arange(h), S)]
                           for o in loc]
                loc_s = loc_s.contiguous().view(T.int16).cpu().numpy().view(np.uint16)
                pr = tp.PartialReduce()
                outs = tp.rowpar_linear_fwd_tp(Xg, Wg.t(), t_local, sel, pr)
                T.cuda.current_stream().synchronize()
                results[g] = ([o.view(T.int16).cpu().numpy().view(np.uint16) for o in outs], loc_s, own)
        except Exception as e:  # pragma: no cover - reported below
            errors.append((g, repr(e)))
            fake.bar.abort()

    threads = [threading.Thread(target=rank_main, args=(g,)) for g in range(P)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    assert caat.device_status() == 0
    Xv, Wv = _round_bf16(X), _round_bf16(W)
    # the processes' local sums on S, folded in process order by the oracle
    sums = np.stack([results[g][1] for g in range(P)])
    red = orc.pcr_bf16(sums, np.arange(S.size, dtype=np.int32))[0][0]
    full, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    notS = np.setdiff1d(np.arange(h), S)
    for g in range(P):
        outs, _, own = results[g]
        for r in range(t_local):
            np.testing.assert_array_equal(outs[r][:, S], red)                 # bit for bit
            np.testing.assert_array_equal(outs[r][:, notS], own[r] if layout == 0 else own[r])
            got = orc.bf16_to_f64(outs[r])
            e = np.linalg.norm(got - full[g * t_local + r]) / np.linalg.norm(full[g * t_local + r])
            assert e <= 1e-2, (g, r, e)
