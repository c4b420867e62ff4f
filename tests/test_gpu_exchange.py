"""GPU parity of the per-GPU steps of the partial channel-reduce across
processes (caat_pcr_pack, caat_rank_fold, caat_pcr_unpack) against the oracle,
bit for bit, and of their composition as the protocol of
partial_activation_sync_gb300.tp runs it (row blocks handed between processes,
folded in process order, gathered and written back), with the processes'
buffers all on this one GPU."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import dev, sel_dev, torch, words

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


def _bits(a, dtype):
    """Host words of float32 values as the device would hold them."""
    return ci.bf16_words(a) if dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _sel_arg(S, by_size):
    return int(S.size) if by_size else sel_dev(S)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,h,ld,p,layout,by_size", [
    (37, 200, 200, 0.5, 0, True),      # contiguous, 16-byte vectors
    (37, 200, 208, 0.5, 0, True),      # strided rows
    (5, 100, 100, 0.27, 0, True),      # |S| = 27: element by element
    (64, 96, 96, 0.5, 1, False),       # random S
    (64, 96, 96, 0.5, 0, False),       # contiguous S as an index list
    (3, 1, 1, 1.0, 0, True),           # one channel
])
def test_pack_unpack_bitexact(caat, dtype, N, h, ld, p, layout, by_size):
    T = torch()
    S = orc.select_channels(h, p, layout, 77)
    Y = ci.normal(7101, (N, ld))
    Yd = dev(Y, dtype)[:, :h]
    P = T.empty((N, S.size), dtype=Yd.dtype, device="cuda")
    caat.pcr_pack(Yd, _sel_arg(S, by_size), P)
    T.cuda.synchronize()
    np.testing.assert_array_equal(words(P), _bits(Y, dtype)[:, S])
    # write back into two outputs whose other channels (and padding) stay untouched
    Pv = ci.normal(7102, (N, S.size))
    Pd = dev(Pv, dtype)
    outs = [dev(ci.normal(7103 + k, (N, ld)), dtype) for k in range(2)]
    before = [words(o) for o in outs]
    caat.pcr_unpack(Pd, _sel_arg(S, by_size), [o[:, :h] for o in outs])
    T.cuda.synchronize()
    for k in range(2):
        want = before[k].copy()
        want[:, S] = _bits(Pv, dtype)
        np.testing.assert_array_equal(words(outs[k]), want)
    assert caat.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("t,rows,cols", [(1, 7, 16), (2, 33, 64), (3, 5, 24), (8, 100, 2048), (4, 9, 13)])
def test_rank_fold_bitexact(caat, dtype, t, rows, cols):
    T = torch()
    R = ci.normal(7201 + t, (t, rows, cols))
    Rd = dev(R, dtype)
    out = T.empty((rows, cols), dtype=Rd.dtype, device="cuda")
    caat.rank_fold(Rd, out)
    T.cuda.synchronize()
    allc = np.arange(cols, dtype=np.int32)
    if dtype == "bf16":
        want = orc.pcr_bf16(ci.bf16_words(R), allc)[0][0]
    else:
        want = orc.pcr_f32(R, allc)[0][0].view(np.uint32)
    np.testing.assert_array_equal(words(out), want)


@pytest.mark.parametrize("procs,t_local,N,h,p,layout", [(2, 4, 37, 256, 0.5, 0), (4, 2, 64, 192, 0.5, 1),
                                                        (8, 1, 100, 512, 0.25, 0)])
def test_exchange_composition_bitexact(caat, procs, t_local, N, h, p, layout):
    """The protocol's steps with every process's buffers on this GPU: pack each
    process's local S sum, cut the dense buffers into `procs` row blocks (what the
    all-to-all delivers), fold block q of all processes in process order, gather
    the folded blocks, and write them back into every local output."""
    T = torch()
    S = orc.select_channels(h, p, layout, 91)
    sel = _sel_arg(S, layout == 0)
    s = S.size
    C = -(-N // procs)
    local = [ci.normal(7300 + g, (t_local, N, h)) for g in range(procs)]
    for g in range(procs):     # the local ranks agree on S (the fused forward wrote their local sum)
        local[g][1:, :, S] = local[g][0][:, S]
    outs = [[dev(local[g][r], "bf16") for r in range(t_local)] for g in range(procs)]
    Ps = []
    for g in range(procs):
        P = T.zeros((procs * C, s), dtype=T.bfloat16, device="cuda")
        caat.pcr_pack(outs[g][0], sel, P[:N])
        Ps.append(P)
    G = T.empty((procs * C, s), dtype=T.bfloat16, device="cuda")
    for q in range(procs):
        R = T.stack([Ps[g][q * C:(q + 1) * C] for g in range(procs)])
        caat.rank_fold(R.contiguous(), G[q * C:(q + 1) * C])
    for g in range(procs):
        caat.pcr_unpack(G[:N], sel, outs[g])
    T.cuda.synchronize()
    sums = np.stack([ci.bf16_words(local[g][0]) for g in range(procs)])
    red = orc.pcr_bf16(sums, S)[0][0]
    notS = np.setdiff1d(np.arange(h), S)
    for g in range(procs):
        for r in range(t_local):
            w = words(outs[g][r])
            np.testing.assert_array_equal(w[:, S], red[:, S])
            np.testing.assert_array_equal(w[:, notS], ci.bf16_words(local[g][r])[:, notS])
    assert caat.device_status() == 0
