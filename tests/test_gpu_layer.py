"""GPU parity of the fused row-parallel layer (forward and backward) against the
CPU oracle (double accumulation).

Tolerances are relative Frobenius errors, max over the t rank outputs, dX and
dW: 1e-5 for fp32 (FFMA, fp32 accumulation) and 1e-2 for bf16 inputs with fp32
accumulation (one bf16 rounding of the output alone is up to 2^-9 relative)."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import TOL, dev, host_values, rel_fro, sel_dev, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


def _weight(Wl32, dtype, layout):
    """Device weight holding logical W [K, h]: 'nn' = stored [h, K] (K contiguous,
    passed as .t()), 'rm' = stored row-major [K, h]."""
    if layout == "nn":
        return dev(np.ascontiguousarray(Wl32.T), dtype).t()
    return dev(Wl32, dtype)


def _fwd_case(caat, t, N, K, h, p, layout_S, dtype, wl="nn", seed=0):
    X = ci.normal(1000 + seed, (N, K))
    Wl = ci.normal(2000 + seed, (K, h), std=0.02)
    S = caat.select_channels(h, p, layout_S, 4000 + seed)
    Xd, Wd = dev(X, dtype), _weight(Wl, dtype, wl)
    outs = caat.rowpar_linear_fwd(Xd, Wd, t, sel_dev(S))
    torch().cuda.synchronize()
    assert caat.device_status() == 0
    got = np.stack([to_f64(o) for o in outs])
    want, _ = orc.rowpar_fwd(host_values(X, dtype), host_values(Wl, dtype), t, S)
    return got, want, S


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t,N,kt,h", [(1, 5, 8, 24), (2, 7, 4, 40), (3, 129, 96, 200),
                                      (8, 33, 16, 72), (4, 64, 24, 130)])
@pytest.mark.parametrize("wl", ["nn", "rm"])
def test_fwd_small_shapes(caat, dtype, t, N, kt, h, wl):
    for p in (0.0, 0.5, 1.0):
        for layout in (0, 1):
            got, want, S = _fwd_case(caat, t, N, kt * t, h, p, layout, dtype, wl, seed=t + N)
            for r in range(t):
                assert rel_fro(got[r], want[r]) <= TOL[dtype], (r, p, layout)
            for r in range(1, t):    # S channels bit-identical across ranks
                assert np.array_equal(got[r][:, S], got[0][:, S])


def test_fwd_zero_k(caat):
    T = torch()
    X = T.zeros((4, 0), device="cuda")
    W = T.zeros((0, 8), device="cuda")
    outs = caat.rowpar_linear_fwd(X, W, 2, sel_dev(np.arange(4)))
    T.cuda.synchronize()
    for o in outs:
        assert bool((o == 0).all())


def _bwd_case(caat, t, N, K, h, p, layout_S, dtype, mode, wl="nn", seed=0, rows=None):
    X = ci.normal(1100 + seed, (N, K))
    Wl = ci.normal(2100 + seed, (K, h), std=0.02)
    G = ci.normal(3100 + seed, (t, N, h))
    S = caat.select_channels(h, p, layout_S, 4100 + seed)
    Xd, Wd = dev(X, dtype), _weight(Wl, dtype, wl)
    Gd = [dev(G[r], dtype) for r in range(t)]
    dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, sel_dev(S), mode)
    torch().cuda.synchronize()
    assert caat.device_status() == 0
    gX, gW = to_f64(dX), to_f64(dW)
    wX, wW = orc.rowpar_bwd(host_values(X, dtype), host_values(Wl, dtype),
                            np.stack([host_values(G[r], dtype) for r in range(t)]), t, S, mode)
    return gX, gW, wX, wW


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("t,N,kt,h", [(1, 5, 8, 24), (2, 7, 4, 40), (3, 129, 96, 200),
                                      (8, 33, 16, 72)])
@pytest.mark.parametrize("wl", ["nn", "rm"])
def test_bwd_small_shapes(caat, dtype, mode, t, N, kt, h, wl):
    for p in (0.0, 0.5, 1.0):
        gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, p, 1, dtype, mode, wl, seed=t + N)
        assert rel_fro(gX, wX) <= TOL[dtype], ("dX", p)
        assert rel_fro(gW, wW) <= TOL[dtype], ("dW", p)


def test_bwd_zero_rows_gives_zero_dw(caat):
    T = torch()
    t, K, h = 2, 8, 16
    X = T.zeros((0, K), device="cuda")
    W = T.randn((h, K), device="cuda").t()
    G = [T.zeros((0, h), device="cuda") for _ in range(t)]
    dX, dW = caat.rowpar_linear_bwd(X, W, G, t, sel_dev(np.arange(4)), 0)
    T.cuda.synchronize()
    assert dX.shape == (0, K) and bool((dW == 0).all())
