"""The library's calls inside a captured CUDA graph: the forward (tile and few-token
kernels), the backward in both placements (its dW chain forks onto a side stream
and joins back through events), the column-parallel backward, and the compact
forward and backward (contiguous S and an index list).  A replay must
give the results of the same calls run eagerly: bit for bit where the kernels fix
the summation order, and within 1e-3 relative Frobenius for dW, whose token-split
parts are added in whatever order they finish."""
import numpy as np
import pytest

import caat_inputs as ci
from tests.gpu_helpers import dev, rel_fro, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


def _capture(T, fn):
    """Warm up on a side stream (torch's rule for capture), then capture fn."""
    s = T.cuda.Stream()
    s.wait_stream(T.cuda.current_stream())
    with T.cuda.stream(s):
        fn()
    T.cuda.current_stream().wait_stream(s)
    T.cuda.synchronize()
    g = T.cuda.CUDAGraph()
    with T.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("N", [256, 8])
def test_rowpar_calls_replay_from_a_graph(caat, N):
    T = torch()
    t, kt, h = 8, 96, 768
    K = t * kt
    X = dev(ci.normal(1501, (N, K)), "bf16")
    W = dev(np.ascontiguousarray(ci.normal(1502, (K, h), std=0.02).T), "bf16").t()
    G = [dev(ci.normal(1503 + r, (N, h)), "bf16") for r in range(t)]
    Y = [T.empty((N, h), dtype=T.bfloat16, device="cuda") for _ in range(t)]
    dX = [T.empty((N, K), dtype=T.bfloat16, device="cuda") for _ in range(2)]
    dW = [T.empty((h, K), dtype=T.bfloat16, device="cuda").t() for _ in range(2)]
    ws = T.empty(caat.rowpar_linear_bwd_workspace(t, N, K, h, 1, 0), dtype=T.uint8, device="cuda")

    def calls():
        caat.rowpar_linear_fwd(X, W, t, h // 2, outs=Y)
        for i, mode in enumerate((caat.CAAT_BWD_REDUCE_DOUT, caat.CAAT_BWD_NO_REDUCE)):
            caat.rowpar_linear_bwd(X, W, G, t, h // 2, mode, dX=dX[i], dW=dW[i], workspace=ws)

    calls()
    T.cuda.synchronize()
    ref = [y.clone() for y in Y] + [x.clone() for x in dX] + [w.clone() for w in dW]
    g = _capture(T, calls)
    for buf in Y + dX + dW:
        buf.zero_()
    g.replay()
    T.cuda.synchronize()
    assert caat.device_status() == 0
    for a, b in zip(Y + dX, ref[: t + 2]):
        assert bool((a.view(T.int16) == b.view(T.int16)).all())
    for a, b in zip(dW, ref[t + 2:]):
        assert rel_fro(to_f64(a), to_f64(b)) <= 1e-3


def test_colpar_backward_replays_from_a_graph(caat):
    T = torch()
    t, N, h, K = 8, 256, 768, 3072
    A = dev(ci.normal(1601, (t, N, h)), "bf16")
    W1 = dev(ci.normal(1602, (h, K), std=0.02), "bf16")
    dZ = dev(ci.normal(1603, (N, K)), "bf16")
    dA = T.empty((t, N, h), dtype=T.bfloat16, device="cuda")
    dW1 = T.empty((h, K), dtype=T.bfloat16, device="cuda")
    ws = T.empty(max(caat.colpar_linear_bwd_workspace(t, N, h, K, 1), 1), dtype=T.uint8, device="cuda")

    def calls():
        caat.colpar_linear_bwd(A, W1, dZ, t, h // 2, dA=dA, dW1=dW1, workspace=ws)

    calls()
    T.cuda.synchronize()
    rA, rW = dA.clone(), dW1.clone()
    g = _capture(T, calls)
    dA.zero_()
    dW1.zero_()
    g.replay()
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert bool((dA.view(T.int16) == rA.view(T.int16)).all())
    assert rel_fro(to_f64(dW1), to_f64(rW)) <= 1e-3


@pytest.mark.parametrize("layout", ["contiguous", "random"])
def test_compact_calls_replay_from_a_graph(caat, layout):
    """The compact forward and backward in a graph: with an index list of S they
    also permute W's rows (and dW's) through the workspace, and the backward's dW
    chain forks onto the side stream before that permute."""
    T = torch()
    from tests.gpu_helpers import sel_dev
    t, N, kt, h = 8, 256, 96, 768
    K = t * kt
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM if layout == "random" else caat.CAAT_S_CONTIGUOUS, 1701)
    sel = sel_dev(S) if layout == "random" else int(S.size)
    ns = int(S.size)
    X = dev(ci.normal(1702, (N, K)), "bf16")
    W = dev(np.ascontiguousarray(ci.normal(1703, (K, h), std=0.02).T), "bf16").t()
    dYS = dev(ci.normal(1704, (N, ns)), "bf16")
    dYN = [dev(ci.normal(1705 + r, (N, h - ns)), "bf16") for r in range(t)]
    YS = T.empty((N, ns), dtype=T.bfloat16, device="cuda")
    YN = [T.empty((N, h - ns), dtype=T.bfloat16, device="cuda") for _ in range(t)]
    dX = T.empty((N, K), dtype=T.bfloat16, device="cuda")
    dW = T.empty((h, K), dtype=T.bfloat16, device="cuda").t()
    idx = layout == "random"
    wsf = T.empty(max(caat.rowpar_linear_compact_workspace(t, N, K, h, 1, idx, False), 1), dtype=T.uint8,
                  device="cuda")
    wsb = T.empty(caat.rowpar_linear_compact_workspace(t, N, K, h, 1, idx, True), dtype=T.uint8, device="cuda")

    def calls():
        caat.rowpar_linear_fwd_compact(X, W, t, sel, YS=YS, YN=YN, workspace=wsf)
        caat.rowpar_linear_bwd_compact(X, W, dYS, dYN, t, sel=sel, dX=dX, dW=dW, workspace=wsb)

    calls()
    T.cuda.synchronize()
    ref = [YS.clone()] + [y.clone() for y in YN] + [dX.clone(), dW.clone()]
    g = _capture(T, calls)
    for buf in [YS] + YN + [dX, dW]:
        buf.zero_()
    g.replay()
    T.cuda.synchronize()
    assert caat.device_status() == 0
    for a, b in zip([YS] + YN + [dX], ref[:-1]):
        assert bool((a.view(T.int16) == b.view(T.int16)).all())
    assert rel_fro(to_f64(dW), to_f64(ref[-1])) <= 1e-3


@pytest.mark.parametrize("N", [1, 8, 64, 200])
@pytest.mark.parametrize("graph", [False, True])
def test_few_token_chain_with_programmatic_launch(caat, N, graph, monkeypatch):
    """The few-token kernel is launched as a programmatic dependent of the
    previous launch (its CTAs may start while that grid finishes; it waits for it
    before touching memory).  A chain of dependent calls -- each call's X is the
    previous call's rank-0 output -- must give the same bits with and without
    that launch mode, one call after another and replayed from a graph.  With
    CAAT_PDL_WEIGHTS=1 the weight tiles of the first ring stages are read before
    the wait: the chain's weights are written by nothing, so that is allowed, and
    X still waits for the call that produced it."""
    T = torch()
    t, h = 8, 512
    K = h
    depth = 6
    Ws = [dev(np.ascontiguousarray(ci.normal(1700 + i, (K, h), std=0.05).T), "bf16").t() for i in range(depth)]
    X0 = dev(ci.normal(1699, (N, K)), "bf16")
    outs = [[T.empty((N, h), dtype=T.bfloat16, device="cuda") for _ in range(t)] for _ in range(depth)]

    def chain():
        x = X0
        for i in range(depth):
            caat.rowpar_linear_fwd(x, Ws[i], t, h // 2, outs=outs[i])
            x = outs[i][0]

    def run():
        for o in outs:
            for y in o:
                y.fill_(float("nan"))
        if graph:
            g = _capture(T, chain)
            for o in outs:
                for y in o:
                    y.fill_(float("nan"))
            g.replay()
        else:
            chain()
        T.cuda.synchronize()
        assert caat.last_kernel() == "rowpar_fwd_skinny_tc" or graph
        return [[y.view(T.int16).cpu().numpy().copy() for y in o] for o in outs]

    monkeypatch.setenv("CAAT_PDL", "0")
    plain = run()
    monkeypatch.setenv("CAAT_PDL", "1")
    pdl = run()
    monkeypatch.setenv("CAAT_PDL_WEIGHTS", "1")
    early_w = run()
    for i in range(depth):
        for r in range(t):
            np.testing.assert_array_equal(pdl[i][r], plain[i][r], err_msg="call %d rank %d" % (i, r))
            np.testing.assert_array_equal(early_w[i][r], plain[i][r], err_msg="weights early: call %d rank %d" % (i, r))
    assert caat.device_status() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("graph", [False, True])
def test_reduce_chain_with_programmatic_launch(caat, dtype, graph, monkeypatch):
    """The standalone reduce is launched as a programmatic dependent of the
    previous launch and waits for it before reading.  A chain of reduces, each
    reading the previous one's outputs (alternating two buffer sets, with a random
    S so that both kinds of channel move), must give the same bits with and
    without that launch mode, one call after another and replayed from a graph."""
    T = torch()
    t, N, h, depth = 4, 256, 768, 6
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 77)
    sel = T.from_numpy(S).cuda()
    src = [dev(ci.normal(2300 + r, (N, h)), dtype) for r in range(t)]
    bufs = [[T.empty_like(src[0]) for _ in range(t)] for _ in range(2)]

    def chain():
        x = src
        for i in range(depth):
            caat.partial_channel_reduce(x, sel, outs=bufs[i % 2])
            x = bufs[i % 2]

    def run():
        for b in bufs:
            for y in b:
                y.fill_(float("nan"))
        if graph:
            g = _capture(T, chain)
            for b in bufs:
                for y in b:
                    y.fill_(float("nan"))
            g.replay()
        else:
            chain()
        T.cuda.synchronize()
        return [[y.view(T.int16 if dtype == "bf16" else T.int32).cpu().numpy().copy() for y in b] for b in bufs]

    monkeypatch.setenv("CAAT_PDL", "0")
    plain = run()
    monkeypatch.setenv("CAAT_PDL", "1")
    pdl = run()
    for j in range(2):
        for r in range(t):
            np.testing.assert_array_equal(pdl[j][r], plain[j][r], err_msg="buffer %d rank %d" % (j, r))
    assert caat.device_status() == 0


@pytest.mark.parametrize("graph", [False, True])
def test_layer_chain_with_programmatic_launch(caat, graph, monkeypatch):
    """The tile forward, the backward GEMMs and the sum of the gradient's S
    channels are launched as programmatic dependents of the previous launch: each
    waits for it before touching memory.  A chain where every call reads what the
    call before it wrote -- forward into the next forward's X, its outputs as the
    backward's gradient, the backward's dX as the next forward's X -- must give the
    same bits with and without that launch mode, in a stream and from a graph.  dW
    is computed in one pass (no accumulator), so it is deterministic too."""
    T = torch()
    t, N, h = 8, 256, 768
    K = h
    depth = 3
    Ws = [dev(np.ascontiguousarray(ci.normal(1800 + i, (K, h), std=0.05).T), "bf16").t() for i in range(depth)]
    X0 = dev(ci.normal(1799, (N, K)), "bf16")
    outs = [[T.empty((N, h), dtype=T.bfloat16, device="cuda") for _ in range(t)] for _ in range(depth)]
    dXs = [T.empty((N, K), dtype=T.bfloat16, device="cuda") for _ in range(depth)]
    dWs = [T.empty((h, K), dtype=T.bfloat16, device="cuda").t() for _ in range(depth)]
    req = (caat.rowpar_linear_bwd_workspace(t, N, K, h, 1, caat.CAAT_BWD_REDUCE_DOUT)
           - caat.rowpar_linear_bwd_workspace(t, N, K, h, 1, caat.CAAT_BWD_NO_REDUCE))
    ws = T.empty(req, dtype=T.uint8, device="cuda")

    def chain():
        x = X0
        for i in range(depth):
            caat.rowpar_linear_fwd(x, Ws[i], t, h // 2, outs=outs[i])
            caat.rowpar_linear_bwd(outs[i][1], Ws[i], outs[i], t, h // 2, caat.CAAT_BWD_REDUCE_DOUT,
                                   dX=dXs[i], dW=dWs[i], workspace=ws)
            x = dXs[i]

    def run():
        bufs = [y for o in outs for y in o] + dXs + dWs
        for b in bufs:
            b.fill_(float("nan"))
        if graph:
            g = _capture(T, chain)
            for b in bufs:
                b.fill_(float("nan"))
            g.replay()
        else:
            chain()
        T.cuda.synchronize()
        return [b.contiguous().view(T.int16).cpu().numpy().copy() for b in bufs]

    monkeypatch.setenv("CAAT_PDL", "0")
    plain = run()
    monkeypatch.setenv("CAAT_PDL", "1")
    pdl = run()
    assert caat.device_status() == 0
    for i, (a, b) in enumerate(zip(pdl, plain)):
        np.testing.assert_array_equal(a, b, err_msg="buffer %d" % i)
