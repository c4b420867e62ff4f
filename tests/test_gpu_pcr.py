"""GPU parity of the standalone partial channel-reduce against the CPU oracle.

The fold order (rank 0..t-1, fp32) is fixed on both sides, so fp32 and bf16
results must match the oracle bit for bit."""
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


def _ref(Y32, dtype, S):
    if dtype == "f32":
        out, red = orc.pcr_f32(Y32, S)
        return out.view(np.uint32), red
    out, red = orc.pcr_bf16(ci.bf16_words(Y32), S)
    return out, red


def _run(caat, Y32, dtype, S, in_place=False, pad=0):
    T = torch()
    t, N, h = Y32.shape
    ins = []
    for r in range(t):
        x = dev(Y32[r], dtype)
        if pad:
            big = T.zeros((N, h + pad), dtype=x.dtype, device="cuda")
            big[:, :h] = x
            x = big[:, :h]
        ins.append(x)
    outs = ins if in_place else None
    outs = caat.partial_channel_reduce(ins, sel_dev(S), outs=outs)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    return np.stack([words(o) for o in outs])


def test_config1_fp32_t2_256x768_bitexact(caat):
    w = ci.WORKLOADS["pcr_f32_t2_256x768"]
    Y = ci.normal(1000 + w.cfg, (w.t, w.N, w.h))
    S = caat.select_channels(w.h, w.p, w.layout)
    assert S.size == 384 and S[0] == 0 and S[-1] == 383
    got = _run(caat, Y, "f32", S)
    want, red = _ref(Y, "f32", S)
    np.testing.assert_array_equal(got, want)
    assert red == w.N * 384
    assert caat.last_kernel() == "pcr_vec"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t", [1, 2, 3, 8, 13])
@pytest.mark.parametrize("N,h", [(1, 8), (7, 40), (129, 768), (33, 1000)])
def test_sweep_bitexact(caat, dtype, t, N, h):
    Y = ci.normal(17 + t + N + h, (t, N, h))
    for p in (0.0, 1.0 / h, 0.5, 1 - 1.0 / h, 1.0):
        for layout in (0, 1):
            S = caat.select_channels(h, p, layout, 4003)
            want, _ = _ref(Y, dtype, S)
            np.testing.assert_array_equal(_run(caat, Y, dtype, S), want)
            np.testing.assert_array_equal(_run(caat, Y, dtype, S, in_place=True), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("h,pad", [(37, 4), (40, 3), (768, 1)])
def test_unaligned_rows_scalar_path(caat, dtype, h, pad):
    t, N = 3, 9
    Y = ci.normal(5 + h, (t, N, h))
    S = caat.select_channels(h, 0.5, 1, 9)
    want, _ = _ref(Y, dtype, S)
    np.testing.assert_array_equal(_run(caat, Y, dtype, S, pad=pad), want)
    assert caat.last_kernel() == "pcr_scalar"


def test_guard_bands_untouched(caat):
    T = torch()
    t, N, h = 4, 33, 200
    Y = ci.normal(77, (t, N, h))
    S = caat.select_channels(h, 0.5, 1, 1)
    ins = [dev(Y[r], "f32") for r in range(t)]
    G = 64
    bufs = [T.full((N * h + 2 * G,), -7.0, device="cuda") for _ in range(t)]
    outs = [b[G:G + N * h].view(N, h) for b in bufs]
    caat.partial_channel_reduce(ins, sel_dev(S), outs=outs)
    T.cuda.synchronize()
    for b in bufs:
        assert bool((b[:G] == -7.0).all()) and bool((b[G + N * h:] == -7.0).all())
    want, _ = _ref(Y, "f32", S)
    np.testing.assert_array_equal(np.stack([words(o) for o in outs]), want)


def test_empty_inputs(caat):
    T = torch()
    for N, h in [(0, 16), (4, 0), (0, 0)]:
        ins = [T.zeros((N, h), device="cuda") for _ in range(2)]
        sel = sel_dev(np.arange(min(h, 3), dtype=np.int32))
        outs = caat.partial_channel_reduce(ins, sel)
        assert [tuple(o.shape) for o in outs] == [(N, h)] * 2


@pytest.mark.parametrize("dtype,t,N,h", [("bf16", 8, 8192, 768), ("f32", 8, 4096, 4096),
                                         ("bf16", 8, 8192, 2048)])
def test_full_size_sampled_rows(caat, dtype, t, N, h):
    # rows are independent: the oracle on a sample of rows gives those rows exactly
    Y = ci.normal(3000 + h, (t, N, h))
    for layout in (0, 1):
        S = caat.select_channels(h, 0.5, layout, 4003)
        got = _run(caat, Y, dtype, S)
        rows = np.random.default_rng(1).choice(N, 16, replace=False)
        rows[0], rows[1] = 0, N - 1
        want, _ = _ref(np.ascontiguousarray(Y[:, rows, :]), dtype, S)
        np.testing.assert_array_equal(got[:, rows, :], want)
        # S channels identical on all ranks, everywhere
        for r in range(1, t):
            np.testing.assert_array_equal(got[r][:, S], got[0][:, S])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t", [16, 32, 64])
def test_maximum_rank_count_bitexact(caat, dtype, t):
    """Up to the largest t the library takes (64): the rank-order fold stays exact."""
    N, h = 19, 136
    Y = ci.normal(23 + t, (t, N, h))
    for p, layout in ((0.5, 0), (0.5, 1), (1.0, 0)):
        S = caat.select_channels(h, p, layout, 4004)
        want, _ = _ref(Y, dtype, S)
        np.testing.assert_array_equal(_run(caat, Y, dtype, S), want)


def test_rank_count_above_maximum_is_rejected(caat):
    T = torch()
    ins = [T.zeros((2, 8), device="cuda") for _ in range(65)]
    with pytest.raises(caat.CaatError):
        caat.partial_channel_reduce(ins, sel_dev(np.arange(4)))
