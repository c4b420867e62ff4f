"""The CUDA-core (FFMA) kernels run bf16 layer work only on request.

bf16 work that no tensor-core kernel takes -- 17 ranks at prefill size, a
row-major weight -- is refused with UNSUPPORTED, before anything is launched,
unless CAAT_ALLOW_FALLBACK=1 is in the environment.  fp32 (no tensor-core path)
and empty work need no opt-in.  The conftest sets the variable for every GPU
test; these tests remove it.  Also here: the other opt-in check of the
arguments, CAAT_CHECK_SEL=1, which validates an index list of S."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import check, dev, host_values, sel_dev, to_f64, torch, words

pytestmark = pytest.mark.gpu

UNSUPPORTED = 2


def _nan_outs(t, N, h, dtype):
    T = torch()
    return [T.full((N, h), float("nan"), dtype=dtype, device="cuda") for _ in range(t)]


def _untouched(ts):
    return all(bool(torch().isnan(x).all()) for x in ts)


def _fwd_want(Xv, Wv, t, S):
    """The oracle's outputs and sum_r |Y_r| on S (an index list of S may fold the
    ranks' rounded partials)."""
    want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    parts, _ = orc.rowpar_fwd(Xv, Wv, t, np.zeros(0, np.int32))
    spread = np.zeros(want.shape[1:])
    spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    return want, spread


@pytest.fixture
def no_opt_in(monkeypatch):
    monkeypatch.delenv("CAAT_ALLOW_FALLBACK", raising=False)


@pytest.mark.parametrize("case", ["t17", "row_major_w"])
def test_bf16_forward_refused_without_opt_in(no_opt_in, monkeypatch, case):
    import partial_activation_sync_gb300 as caat
    T = torch()
    if case == "t17":
        t, N, K, h = 17, 256, 17 * 64, 256
    else:
        t, N, K, h = 8, 256, 1024, 384
    X = ci.normal(3, (N, K))
    Wl = ci.normal(4, (K, h), std=0.02)
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 5)
    sel = sel_dev(S)
    Xd = dev(X, "bf16")
    if case == "t17":
        Wd = dev(np.ascontiguousarray(Wl.T), "bf16").t()     # nn.Linear layout
    else:
        Wd = dev(Wl, "bf16")                                 # row-major [K, h]
    outs = _nan_outs(t, N, h, T.bfloat16)
    n0 = caat.launch_count()
    with pytest.raises(caat.CaatError) as e:
        caat.rowpar_linear_fwd(Xd, Wd, t, sel, outs=outs)
    assert e.value.status == UNSUPPORTED
    T.cuda.synchronize()
    assert caat.launch_count() == n0, "a refused call launched a kernel"
    assert _untouched(outs)

    # the same call with the opt-in runs on the CUDA cores and matches the oracle
    monkeypatch.setenv("CAAT_ALLOW_FALLBACK", "1")
    caat.rowpar_linear_fwd(Xd, Wd, t, sel, outs=outs)
    T.cuda.synchronize()
    assert caat.last_kernel() == "rowpar_fwd_simt"
    want, spread = _fwd_want(host_values(X, "bf16"), host_values(Wl, "bf16"), t, S)
    for r in range(t):
        check(to_f64(outs[r]), want[r], "bf16", what=r, spread=spread)


def test_fp32_and_empty_work_need_no_opt_in(no_opt_in):
    import partial_activation_sync_gb300 as caat
    T = torch()
    t, N, K, h = 17, 64, 17 * 16, 96
    X = ci.normal(6, (N, K))
    Wl = ci.normal(7, (K, h), std=0.05)
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 8)
    outs = caat.rowpar_linear_fwd(dev(X, "f32"), dev(Wl, "f32"), t, sel_dev(S))
    T.cuda.synchronize()
    want, spread = _fwd_want(host_values(X, "f32"), host_values(Wl, "f32"), t, S)
    for r in range(t):
        check(to_f64(outs[r]), want[r], "f32", what=r, spread=spread)
    # K = 0 in bf16: an empty sum, zeros, no opt-in needed
    Xe = T.zeros((N, 0), dtype=T.bfloat16, device="cuda")
    We = T.zeros((0, h), dtype=T.bfloat16, device="cuda")
    oe = caat.rowpar_linear_fwd(Xe, We, 4, sel_dev(S), outs=_nan_outs(4, N, h, T.bfloat16))
    T.cuda.synchronize()
    assert all(int(np.count_nonzero(words(o))) == 0 for o in oe)


def test_bf16_backward_refused_before_the_reduce(no_opt_in, monkeypatch):
    """A row-major weight in the backward: refused before the reduce of dOut is
    launched, dX, dW and the workspace untouched."""
    import partial_activation_sync_gb300 as caat
    T = torch()
    t, N, K, h = 4, 128, 512, 256
    X = ci.normal(9, (N, K))
    Wl = ci.normal(10, (K, h), std=0.02)
    G = ci.normal(11, (t, N, h))
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 12)
    Xd, Wd = dev(X, "bf16"), dev(Wl, "bf16")
    Gd = [dev(G[r], "bf16") for r in range(t)]
    dX = T.full((N, K), float("nan"), dtype=T.bfloat16, device="cuda")
    dW = T.full((K, h), float("nan"), dtype=T.bfloat16, device="cuda")
    need = caat.rowpar_linear_bwd_workspace(t, N, K, h, caat.CAAT_BF16, caat.CAAT_BWD_REDUCE_DOUT)
    ws = T.full((need,), 0xA5, dtype=T.uint8, device="cuda")
    n0 = caat.launch_count()
    with pytest.raises(caat.CaatError) as e:
        caat.rowpar_linear_bwd(Xd, Wd, Gd, t, sel_dev(S), caat.CAAT_BWD_REDUCE_DOUT, dX=dX, dW=dW, workspace=ws)
    assert e.value.status == UNSUPPORTED
    T.cuda.synchronize()
    assert caat.launch_count() == n0
    assert _untouched([dX, dW])
    assert bool((ws == 0xA5).all())

    monkeypatch.setenv("CAAT_ALLOW_FALLBACK", "1")
    caat.rowpar_linear_bwd(Xd, Wd, Gd, t, sel_dev(S), caat.CAAT_BWD_REDUCE_DOUT, dX=dX, dW=dW, workspace=ws)
    T.cuda.synchronize()
    want_dX, want_dW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                                      host_values(G, "bf16"), t, S, orc.REDUCE_DOUT)
    check(to_f64(dX), want_dX, "bf16", bwd=True, what="dX")
    check(to_f64(dW), want_dW, "bf16", bwd=True, what="dW")


def test_tensor_core_shapes_need_no_opt_in(no_opt_in):
    """The layer shapes the tensor-core kernels take run without the variable."""
    import partial_activation_sync_gb300 as caat
    T = torch()
    t, N, K, h = 8, 256, 1024, 512
    X = ci.normal(13, (N, K))
    Wl = ci.normal(14, (K, h), std=0.02)
    G = ci.normal(15, (t, N, h))
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 16)
    Xd = dev(X, "bf16")
    Wd = dev(np.ascontiguousarray(Wl.T), "bf16").t()
    caat.rowpar_linear_fwd(Xd, Wd, t, sel_dev(S))
    assert caat.last_kernel() != "rowpar_fwd_simt"
    caat.rowpar_linear_bwd(Xd, Wd, [dev(G[r], "bf16") for r in range(t)], t, sel_dev(S))
    assert caat.last_kernel() != "batched_gemm_simt"
    T.cuda.synchronize()
    assert caat.device_status() == 0


@pytest.mark.parametrize("bad", ["duplicate", "unsorted", "out_of_range"])
def test_index_list_debug_check(bad, monkeypatch):
    """CAAT_CHECK_SEL=1 validates an index list of S on the host (ascending,
    unique, inside [0, h)) before anything is launched; a valid list passes."""
    import partial_activation_sync_gb300 as caat
    T = torch()
    t, N, K, h = 4, 128, 256, 256
    X = dev(ci.normal(21, (N, K)), "bf16")
    Wd = dev(np.ascontiguousarray(ci.normal(22, (K, h), std=0.02).T), "bf16").t()
    S = np.arange(0, h, 2, dtype=np.int32)
    if bad == "duplicate":
        S[5] = S[4]
    elif bad == "unsorted":
        S[[3, 4]] = S[[4, 3]]
    else:
        S[-1] = h
    monkeypatch.setenv("CAAT_CHECK_SEL", "1")
    outs = _nan_outs(t, N, h, T.bfloat16)
    n0 = caat.launch_count()
    with pytest.raises(caat.CaatError) as e:
        caat.rowpar_linear_fwd(X, Wd, t, sel_dev(S), outs=outs)
    assert e.value.status == 1                       # CAAT_ERR_INVALID_ARG
    with pytest.raises(caat.CaatError) as e:
        caat.partial_channel_reduce(outs, sel_dev(S))
    assert e.value.status == 1
    T.cuda.synchronize()
    assert caat.launch_count() == n0 and _untouched(outs)
    good = np.arange(0, h, 2, dtype=np.int32)
    caat.rowpar_linear_fwd(X, Wd, t, sel_dev(good), outs=outs)
    T.cuda.synchronize()
    assert caat.device_status() == 0
