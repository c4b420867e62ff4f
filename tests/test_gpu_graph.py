"""The library's calls inside a captured CUDA graph: the forward (tile and few-token
kernels), the backward in both placements (its dW chain forks onto a side stream
and joins back through events), and the column-parallel backward.  A replay must
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
