"""GPU parity of the compact outputs (the S channels stored once, YS, and each
rank's other channels, YN[r]) and of their backward.

Each case is checked twice:
  * against the oracle: YS = the S channels of any rank's output, YN[r] = rank r's
    other channels; the backward against the oracle's reduce-dOut backward of a
    gradient whose S channels sum over the ranks to dYS (rank 0 carries dYS, the
    others zero) and whose other channels are dYN[r];
  * bit for bit against the library's plain form of the same call (the same tiles
    and sums, written to a different layout), so the compact routing neither
    drops, moves nor re-rounds anything.
Shapes cover 192- and 256-wide tiles, CTA pairs, a tile that straddles the end of
S (MIXED: its S chunks are written only after the last shard), t = 1, S empty,
S = every channel, ragged rows and a ragged last channel chunk, and output row
strides wider than the rows (the padding must stay untouched)."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import check, dev, host_values, to_f64, torch, words

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


def _w_nn(Wl):
    """logical W [K, h] stored as an nn.Linear weight [h, K] (passed as .t())."""
    return dev(np.ascontiguousarray(Wl.T), "bf16").t()


def _padded(N, cols, pad):
    """A [N, cols] view of a NaN-filled [N, cols + pad] bf16 buffer."""
    T = torch()
    buf = T.full((N, cols + pad), float("nan"), dtype=T.bfloat16, device="cuda")
    return buf, buf[:, :cols]


# (t, N, k_t, h, n_sel, note)
FWD_SHAPES = [
    (8, 300, 96, 768, 384, "192-wide tiles, ragged rows"),
    (8, 256, 128, 768, 320, "256-wide tiles, a MIXED tile"),
    (4, 512, 512, 1024, 512, "CTA pairs"),
    (4, 512, 512, 1024, 448, "CTA pairs, a MIXED tile"),
    (1, 256, 256, 512, 256, "t = 1"),
    (8, 256, 64, 512, 0, "S empty"),
    (8, 256, 64, 512, 512, "S = every channel"),
    (2, 200, 64, 328, 128, "ragged last channel chunk"),
]


@pytest.mark.parametrize("t,N,kt,h,n_sel,note", FWD_SHAPES)
def test_fwd_compact_parity(caat, t, N, kt, h, n_sel, note, monkeypatch):
    T = torch()
    K = kt * t
    seed = t * 7 + N + h + n_sel
    X = ci.normal(1000 + seed, (N, K))
    Wl = ci.normal(2000 + seed, (K, h), std=0.02)
    Xd, Wd = dev(X, "bf16"), _w_nn(Wl)
    ys_buf, YS = _padded(N, n_sel, 24)
    yn = [_padded(N, h - n_sel, 40) for _ in range(t)]
    YN = [v for _, v in yn]
    caat.rowpar_linear_fwd_compact(Xd, Wd, t, n_sel, YS=YS, YN=YN)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert caat.last_kernel() == "rowpar_fwd_tc"
    # padding columns untouched
    assert bool(T.isnan(ys_buf[:, n_sel:]).all())
    for buf, _ in yn:
        assert bool(T.isnan(buf[:, h - n_sel:]).all())
    S = np.arange(n_sel, dtype=np.int32)
    want, _ = orc.rowpar_fwd(host_values(X, "bf16"), host_values(Wl, "bf16"), t, S)
    if n_sel > 0:
        check(to_f64(YS), want[0][:, :n_sel], "bf16", what=("YS", note))
    for r in range(t):
        if h > n_sel:
            check(to_f64(YN[r]), want[r][:, n_sel:], "bf16", what=("YN", r, note))
    # the plain form of the same call on the same tile kernel: the same bits, laid
    # out per rank (up to 256 tokens the plain form takes the few-token kernel,
    # which sums S in another order)
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")
    full = caat.rowpar_linear_fwd(Xd, Wd, t, n_sel)
    T.cuda.synchronize()
    for r in range(t):
        fw = words(full[r])
        if n_sel > 0:
            assert np.array_equal(words(YS), fw[:, :n_sel]), (note, r)
        if h > n_sel:
            assert np.array_equal(words(YN[r]), fw[:, n_sel:]), (note, r)


def test_fwd_compact_declines(caat):
    """An n_sel that is not a multiple of 64, and a token count the tile kernel does
    not take (the few-token kernels have no compact form): UNSUPPORTED, nothing
    launched."""
    T = torch()
    t, K, h = 4, 256, 512
    for N, n_sel in ((256, 100), (8, 256)):
        X = dev(ci.normal(3, (N, K)), "bf16")
        Wd = _w_nn(ci.normal(4, (K, h), std=0.02))
        n0 = caat.launch_count()
        with pytest.raises(caat.CaatError) as e:
            caat.rowpar_linear_fwd_compact(X, Wd, t, n_sel)
        assert e.value.status == 2
        T.cuda.synchronize()
        assert caat.launch_count() == n0


# (t, N, k_t, h, n_sel, note)
BWD_SHAPES = [
    (8, 256, 96, 768, 384, "130M-like"),
    (4, 300, 256, 512, 128, "ragged rows"),
    (2, 512, 512, 1024, 512, "CTA pairs"),
    (2, 256, 512, 1024, 0, "S empty"),
    (2, 256, 256, 512, 512, "S = every channel"),
]


def _required_ws(caat, t, N, K, h, n_sel):
    """A workspace holding only what the plain backward requires (the reduced
    gradient, when it reduces): no room for the dW accumulator, so dW is not split."""
    T = torch()
    req = 0
    if n_sel > 0 and t > 1:
        req = (caat.rowpar_linear_bwd_workspace(t, N, K, h, caat.CAAT_BF16, caat.CAAT_BWD_REDUCE_DOUT)
               - caat.rowpar_linear_bwd_workspace(t, N, K, h, caat.CAAT_BF16, caat.CAAT_BWD_NO_REDUCE))
    return T.empty(req, dtype=T.uint8, device="cuda")


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("t,N,kt,h,n_sel,note", BWD_SHAPES)
def test_bwd_compact_parity(caat, t, N, kt, h, n_sel, note, split):
    """split: the fp32 dW accumulator given (dW reduced over tokens in several
    parts, whose fp32 adds land in no fixed order) or not (one pass, deterministic:
    then dW too is compared bit for bit with the plain form)."""
    T = torch()
    K = kt * t
    seed = t * 5 + N + h + n_sel
    X = ci.normal(1100 + seed, (N, K))
    Wl = ci.normal(2100 + seed, (K, h), std=0.02)
    GS = ci.normal(3100 + seed, (N, n_sel))
    GN = ci.normal(3200 + seed, (t, N, h - n_sel))
    Xd, Wd = dev(X, "bf16"), _w_nn(Wl)
    dYS = dev(GS, "bf16")
    dYN = [dev(GN[r], "bf16") for r in range(t)]
    ws = None if split else T.empty(0, dtype=T.uint8, device="cuda")
    dX, dW = caat.rowpar_linear_bwd_compact(Xd, Wd, dYS, dYN, t, workspace=ws)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    # the oracle: rank 0's gradient carries dYS on S, the other ranks zero there
    G = np.zeros((t, N, h))
    G[0][:, :n_sel] = host_values(GS, "bf16")
    for r in range(t):
        G[r][:, n_sel:] = host_values(GN[r], "bf16")
    S = np.arange(n_sel, dtype=np.int32)
    wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"), G, t, S, orc.REDUCE_DOUT)
    check(to_f64(dX), wX, "bf16", bwd=True, what=("dX", note))
    check(to_f64(dW), wW, "bf16", bwd=True, what=("dW", note))
    # the plain form with that gradient: its sum over S is exactly dYS, so the
    # same GEMMs see the same operands
    Gd = [dev(G[r].astype(np.float32), "bf16") for r in range(t)]
    pX, pW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, n_sel, caat.CAAT_BWD_REDUCE_DOUT,
                                    workspace=None if split else _required_ws(caat, t, N, K, h, n_sel))
    T.cuda.synchronize()
    assert np.array_equal(words(dX), words(pX)), note
    if not split:
        assert np.array_equal(words(dW.t()), words(pW.t())), note


@pytest.mark.parametrize("wname,li", [("7b_prefill", 0), ("7b_prefill", 1), ("130m", 0), ("130m", 1)])
def test_compact_full_size_matches_plain_form(caat, wname, li):
    """At the benchmark's shapes (p = 0.5, contiguous S): the compact forward gives
    the plain form's bits, and the compact backward (the S gradient summed once)
    the plain reduce-dOut backward's."""
    T = torch()
    w = ci.WORKLOADS[wname]
    L = w.layers[li]
    n_sel = int(caat.select_channels(w.h, w.p).size)
    g = T.Generator(device="cuda").manual_seed(11 + li)
    X = T.randn((w.N, L.K), device="cuda", generator=g).to(T.bfloat16)
    Wd = (T.randn((w.h, L.K), device="cuda", generator=g) * 0.02).to(T.bfloat16).t()
    YS, YN = caat.rowpar_linear_fwd_compact(X, Wd, w.t, n_sel)
    full = caat.rowpar_linear_fwd(X, Wd, w.t, n_sel)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    for r in range(w.t):
        assert T.equal(YS, full[r][:, :n_sel]) and T.equal(YN[r], full[r][:, n_sel:]), r
    del full, YN
    if not w.backward:
        return
    dYS = T.randn((w.N, n_sel), device="cuda", generator=g).to(T.bfloat16)
    dYN = [T.randn((w.N, w.h - n_sel), device="cuda", generator=g).to(T.bfloat16) for _ in range(w.t)]
    # dW in one pass (no accumulator: a split's fp32 adds land in no fixed order)
    dX, dW = caat.rowpar_linear_bwd_compact(X, Wd, dYS, dYN, w.t,
                                            workspace=T.empty(0, dtype=T.uint8, device="cuda"))
    G = [T.cat([dYS if r == 0 else T.zeros_like(dYS), dYN[r]], dim=1) for r in range(w.t)]
    pX, pW = caat.rowpar_linear_bwd(X, Wd, G, w.t, n_sel, caat.CAAT_BWD_REDUCE_DOUT,
                                    workspace=_required_ws(caat, w.t, w.N, L.K, w.h, n_sel))
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert T.equal(dX, pX) and T.equal(dW, pW)


# (t, N, k_t, h, p, note): a seeded random S of |S| = p h channels (a multiple of 64)
RANDOM_SHAPES = [
    (8, 300, 96, 768, 0.5, "130M-like, 192-wide tiles"),
    (4, 512, 512, 1024, 0.5, "CTA pairs"),
    (2, 256, 256, 512, 0.25, "p = 1/4"),
]


@pytest.mark.parametrize("t,N,kt,h,p,note", RANDOM_SHAPES)
def test_random_set_compact_parity(caat, t, N, kt, h, p, note):
    """An index list of S: YS holds S's channels in ascending order and YN[r] the
    other channels of rank r.  Against the oracle, and bit for bit against the
    contiguous compact call on W with its channels renamed S-first (what the
    index-list call runs internally); the backward likewise (dX bit for bit, dW
    through the accumulator, whose rows return to channel order)."""
    from tests.gpu_helpers import sel_dev
    T = torch()
    K = kt * t
    seed = 17 * t + N + h
    S = caat.select_channels(h, p, caat.CAAT_S_RANDOM, 4000 + seed)
    assert 0 < S.size < h and S.size % 64 == 0
    U = np.setdiff1d(np.arange(h), S)
    perm = np.concatenate([S, U])
    X = ci.normal(1000 + seed, (N, K))
    Wl = ci.normal(2000 + seed, (K, h), std=0.02)
    Xd, Wd = dev(X, "bf16"), _w_nn(Wl)
    Xv, Wv = host_values(X, "bf16"), host_values(Wl, "bf16")
    YS, YN = caat.rowpar_linear_fwd_compact(Xd, Wd, t, sel_dev(S))
    T.cuda.synchronize()
    assert caat.device_status() == 0
    want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    check(to_f64(YS), want[0][:, S], "bf16", what=("YS", note))
    for r in range(t):
        check(to_f64(YN[r]), want[r][:, U], "bf16", what=("YN", r, note))
    Wp = _w_nn(Wl[:, perm])
    cS, cN = caat.rowpar_linear_fwd_compact(Xd, Wp, t, int(S.size))
    T.cuda.synchronize()
    assert T.equal(YS, cS) and all(T.equal(a, b) for a, b in zip(YN, cN)), note
    # backward
    GS = ci.normal(3100 + seed, (N, S.size))
    GN = ci.normal(3200 + seed, (t, N, U.size))
    dYS = dev(GS, "bf16")
    dYN = [dev(GN[r], "bf16") for r in range(t)]
    G = np.zeros((t, N, h))
    G[0][:, S] = host_values(GS, "bf16")
    for r in range(t):
        G[r][:, U] = host_values(GN[r], "bf16")
    wX, wW = orc.rowpar_bwd(Xv, Wv, G, t, S, orc.REDUCE_DOUT)
    pX, pW = caat.rowpar_linear_bwd_compact(Xd, Wp, dYS, dYN, t,
                                            workspace=T.empty(0, dtype=T.uint8, device="cuda"))
    full = caat.rowpar_linear_compact_workspace(t, N, K, h, caat.CAAT_BF16, True, True)
    required = full - caat.rowpar_linear_compact_workspace(t, N, K, h, caat.CAAT_BF16, False, True)
    # with the fp32 accumulator (dW may be split over tokens: rows back to channel
    # order as it is rounded), and with only the required part (dW staged in the
    # S-first order, then its rows moved back)
    for ws_bytes in (full, required):
        ws = T.empty(ws_bytes, dtype=T.uint8, device="cuda")
        dX, dW = caat.rowpar_linear_bwd_compact(Xd, Wd, dYS, dYN, t, sel=sel_dev(S), workspace=ws)
        T.cuda.synchronize()
        assert caat.device_status() == 0
        check(to_f64(dX), wX, "bf16", bwd=True, what=("dX", note, ws_bytes))
        check(to_f64(dW), wW, "bf16", bwd=True, what=("dW", note, ws_bytes))
        assert T.equal(dX, pX), note
        if ws_bytes == required:
            # one pass over the tokens on the renamed W, rows moved back: the same bits
            assert T.equal(dW.t()[T.from_numpy(perm).cuda()], pW.t()), note


def test_random_set_compact_declines_short_workspace(caat):
    """An index list without room for the permuted W: INVALID_ARG, nothing launched."""
    from tests.gpu_helpers import sel_dev
    T = torch()
    t, N, K, h = 4, 256, 256, 512
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 3)
    X = dev(ci.normal(5, (N, K)), "bf16")
    Wd = _w_nn(ci.normal(6, (K, h), std=0.02))
    small = T.empty(1024, dtype=T.uint8, device="cuda")
    n0 = caat.launch_count()
    with pytest.raises(caat.CaatError) as e:
        caat.rowpar_linear_fwd_compact(X, Wd, t, sel_dev(S), workspace=small)
    assert e.value.status == 1
    T.cuda.synchronize()
    assert caat.launch_count() == n0
