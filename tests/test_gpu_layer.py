"""GPU parity of the fused row-parallel layer (forward and backward) against the
CPU oracle (double accumulation).

Tolerances are relative Frobenius errors, max over the t rank outputs, dX and
dW: 1e-5 for fp32 (FFMA, fp32 accumulation) and 1e-2 for bf16 inputs with fp32
accumulation (one bf16 rounding of the output alone is up to 2^-9 relative)."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import check, dev, host_values, sel_dev, to_f64, torch

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


def _spread(Xv, Wv, t, S):
    """sum_r |Y_r| on the channels of S (zero elsewhere): the scale of the rounding
    of the ranks' partials when the S channels fold them after rounding."""
    parts, _ = orc.rowpar_fwd(Xv, Wv, t, np.zeros(0, np.int32))
    spread = np.zeros(parts.shape[1:])
    spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    return spread


# oracle results by case: the same case runs under several kernel modes
_ORACLE_CACHE = {}
_ORACLE_CACHE_BYTES = [0]


def _oracle_fwd(key, Xv, Wv, t, S):
    if key in _ORACLE_CACHE:
        return _ORACLE_CACHE[key]
    want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    if _ORACLE_CACHE_BYTES[0] + want.nbytes > (1 << 30):
        _ORACLE_CACHE.clear()
        _ORACLE_CACHE_BYTES[0] = 0
    _ORACLE_CACHE[key] = want
    _ORACLE_CACHE_BYTES[0] += want.nbytes
    return want


def _fwd_case(caat, t, N, K, h, p, layout_S, dtype, wl="nn", seed=0, by_size=False):
    """by_size: a contiguous S passed by its size (the null index list), which is
    what lets the tile kernel cut its NO_S tiles into per-shard pieces."""
    X = ci.normal(1000 + seed, (N, K))
    Wl = ci.normal(2000 + seed, (K, h), std=0.02)
    S = caat.select_channels(h, p, layout_S, 4000 + seed)
    Xd, Wd = dev(X, dtype), _weight(Wl, dtype, wl)
    outs = caat.rowpar_linear_fwd(Xd, Wd, t, int(S.size) if by_size else sel_dev(S))
    torch().cuda.synchronize()
    assert caat.device_status() == 0
    got = np.stack([to_f64(o) for o in outs])
    Xv, Wv = host_values(X, dtype), host_values(Wl, dtype)
    want = _oracle_fwd((t, N, K, h, S.tobytes(), dtype, seed), Xv, Wv, t, S)
    spread = None
    if not by_size and 0 < S.size < h and t > 1:
        # an index list of S: the S channels fold the ranks' rounded partials
        parts = _oracle_fwd((t, N, K, h, b"", dtype, seed), Xv, Wv, t, np.zeros(0, np.int32))
        spread = np.zeros((N, h))
        spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    return got, want, S, spread


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t,N,kt,h", [(1, 5, 8, 24), (2, 7, 4, 40), (3, 129, 96, 200),
                                      (8, 33, 16, 72), (4, 64, 24, 130)])
@pytest.mark.parametrize("wl", ["nn", "rm"])
def test_fwd_small_shapes(caat, dtype, t, N, kt, h, wl):
    for p in (0.0, 0.5, 1.0):
        for layout in (0, 1):
            got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, layout, dtype, wl, seed=t + N)
            for r in range(t):
                check(got[r], want[r], dtype, what=(r, p, layout), spread=spread)
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
        check(gX, wX, dtype, bwd=True, what=("dX", p))
        check(gW, wW, dtype, bwd=True, what=("dW", p))


def test_bwd_zero_rows_gives_zero_dw(caat):
    T = torch()
    t, K, h = 2, 8, 16
    X = T.zeros((0, K), device="cuda")
    W = T.randn((h, K), device="cuda").t()
    G = [T.zeros((0, h), device="cuda") for _ in range(t)]
    dX, dW = caat.rowpar_linear_bwd(X, W, G, t, sel_dev(np.arange(4)), 0)
    T.cuda.synchronize()
    assert dX.shape == (0, K) and bool((dW == 0).all())


# ------------------------------------------------ tensor-core (tcgen05) path

TC_SHAPES = [
    # t, N, k_t, h    -- ragged rows (N % 128), ragged channels (h % 256), k_t % 64
    (2, 300, 64, 264),
    (8, 256, 96, 768),
    (3, 129, 200, 520),
    (1, 128, 128, 256),
    (8, 384, 344, 512),
    (5, 640, 72, 1032),
    (3, 700, 64, 520),      # six row blocks: three CTA pairs, ragged last block
]
# the forward also takes h = 192 (one 192-wide tile; the backward kernels need h >= 256)
TC_FWD_SHAPES = TC_SHAPES + [
    (4, 200, 64, 192),      # the smallest h: one 192-wide tile
    (3, 260, 128, 576),     # 192-wide tiles: three per row block
    (2, 300, 256, 384),     # 192-wide tiles with shards of 4 k-blocks: the deeper ring
    (16, 256, 64, 512),     # the most ranks the tile kernel takes (one tensor map each)
]


@pytest.fixture(params=["2", "1", "1/192", "2/192", "1:m", "2:m", "1/192:m", "2:r", "1/192:r", "2:f", "1:f"])
def fwd_mode(request, monkeypatch):
    """Cluster shape of the forward: 2 = one CTA pair (cta_group::2, 256-row
    tiles; the default for long shards from two row blocks up), 1 = one CTA per
    128 x 256 tile; "/192": the same with 192-channel tiles (where h is a
    multiple of 192)."""
    # ":m": row-block-major work order; ":r": every tile whole, in rounds (no
    # per-shard pieces of NO_S tiles); ":f": whole tiles first, pieces after
    mode, _, opt = request.param.partition(":")
    cl, _, bn = mode.partition("/")
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")      # the tile kernel at any token count
    monkeypatch.setenv("CAAT_FWD_CLUSTER", cl)
    monkeypatch.setenv("CAAT_FWD_BN", bn or "256")
    monkeypatch.setenv("CAAT_FWD_ORDER", "m" if opt == "m" else "n")
    monkeypatch.setenv("CAAT_FWD_SCHED", {"r": "rounds", "f": "first"}.get(opt, "interleaved"))
    return request.param


@pytest.mark.parametrize("t,N,kt,h", TC_FWD_SHAPES)
def test_fwd_tc_parity(caat, t, N, kt, h, fwd_mode, monkeypatch):
    # the tile kernel, also at N <= 256 where the few-token kernel would run
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")
    # p = 1/h and 1 - 1/h: a single channel in S, a single channel outside it
    for p in (0.0, 1.0 / h, 0.25, 0.5, 0.75, 1.0 - 1.0 / h, 1.0):
        # contiguous S by size (balanced schedule) and as an index list; random S
        for layout, by_size in ((0, True), (0, False), (1, False)):
            got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, layout, "bf16", "nn", seed=7 * t + h,
                                     by_size=by_size)
            assert caat.last_kernel() == "rowpar_fwd_tc"
            for r in range(t):
                check(got[r], want[r], "bf16", what=(r, p, layout), spread=spread)
            for r in range(1, t):
                assert np.array_equal(got[r][:, S], got[0][:, S])


def test_fwd_tc_boundary_tile_mixed(caat, fwd_mode):
    # |S| = 300 with contiguous S: tile 0 all in S, tile 1 mixed, tile 2 outside
    t, N, kt, h = 4, 256, 64, 768
    X = ci.normal(901, (N, kt * t))
    Wl = ci.normal(902, (kt * t, h), std=0.02)
    S = np.arange(300, dtype=np.int32)
    outs = caat.rowpar_linear_fwd(dev(X, "bf16"), _weight(Wl, "bf16", "nn"), t, sel_dev(S))
    torch().cuda.synchronize()
    assert caat.last_kernel() == "rowpar_fwd_tc"
    got = np.stack([to_f64(o) for o in outs])
    Xv, Wv = host_values(X, "bf16"), host_values(Wl, "bf16")
    want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    # an index list of S: the S channels fold the ranks' rounded partials (except
    # in the MIXED-tile mode of the ":r" schedule, where this bound is just looser)
    parts, _ = orc.rowpar_fwd(Xv, Wv, t, np.zeros(0, np.int32))
    spread = np.zeros((N, h))
    spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    for r in range(t):
        check(got[r], want[r], "bf16", spread=spread)
        # per-column check: the non-S half of the mixed tile is this rank's own sum
        check(got[r][:, 300:512], want[r][:, 300:512], "bf16")


def test_fwd_tc_output_guard(caat, fwd_mode):
    # outputs with a row stride wider than h: the padding must stay untouched
    T = torch()
    t, N, kt, h, ld = 2, 200, 64, 256, 264
    X = ci.normal(903, (N, kt * t))
    Wl = ci.normal(904, (kt * t, h), std=0.02)
    S = caat.select_channels(h, 0.5, 1, 5)
    bufs = [T.full((N, ld), 7.0, dtype=T.bfloat16, device="cuda") for _ in range(t)]
    outs = [b[:, :h] for b in bufs]
    caat.rowpar_linear_fwd(dev(X, "bf16"), _weight(Wl, "bf16", "nn"), t, sel_dev(S), outs=outs)
    T.cuda.synchronize()
    assert caat.last_kernel() == "rowpar_fwd_tc"
    for b in bufs:
        assert bool((b[:, h:] == 7.0).all())
    Xv, Wv = host_values(X, "bf16"), host_values(Wl, "bf16")
    want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
    spread = _spread(Xv, Wv, t, S)
    for r in range(t):
        check(to_f64(outs[r]), want[r], "bf16", spread=spread)


FULL = [("130m", 0), ("130m", 1), ("1.1b", 0), ("1.1b", 1), ("7b_prefill", 0), ("7b_prefill", 1)]


def _block_samples(n, block, seed):
    """One index drawn in every block of `block` consecutive indices of range(n),
    plus the first and the last index: every tile along that dimension is hit."""
    rng = np.random.default_rng(seed)
    idx = [min(b0 + int(rng.integers(0, block)), n - 1) for b0 in range(0, n, block)]
    return np.unique(np.array(idx + [0, n - 1], dtype=np.int64))


def _bench_sel(S, layout):
    """S as the benchmark passes it: a contiguous S by its size (null index list),
    a random one as a device index tensor."""
    return int(S.size) if layout == 0 else sel_dev(S)


@pytest.mark.parametrize("wname,li", FULL)
def test_fwd_full_size_sampled_rows(caat, wname, li):
    """Full workload sizes in the benchmark's launch configuration (contiguous S
    passed by its size, as the benchmark does).  Rows are independent, so the
    oracle on one sampled row of every 128-row block gives those rows exactly; all
    channels of those rows are checked, so every output tile is reached."""
    w = ci.WORKLOADS[wname]
    X, Wl, _ = ci.layer_tensors(w, li)
    ps = (0.0, 0.25, 0.5, 0.75, 1.0) if wname == "1.1b" else (w.p,)
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    rows = _block_samples(w.N, 128, li)
    Xs = host_values(X[rows], "bf16")
    Wv = host_values(Wl, "bf16")
    for p in ps:
        for layout in (0, 1):
            S = caat.select_channels(w.h, p, layout, w.seeds()["perm"])
            outs = caat.rowpar_linear_fwd(Xd, Wd, w.t, _bench_sel(S, layout))
            torch().cuda.synchronize()
            assert caat.device_status() == 0
            assert caat.last_kernel() == "rowpar_fwd_tc"
            want, _ = orc.rowpar_fwd(Xs, Wv, w.t, S)
            spread = None
            if layout == 1 and 0 < S.size < w.h:
                # a random S (index list): the S channels fold the rounded partials
                parts, _ = orc.rowpar_fwd(Xs, Wv, w.t, np.zeros(0, np.int32))
                spread = np.zeros(want.shape[1:])
                spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
            for r in range(w.t):
                got = to_f64(outs[r][rows.tolist()])
                check(got, want[r], "bf16", what=(p, layout, r), spread=spread)
            full0 = outs[0][:, S.tolist()] if S.size else None
            for r in range(1, w.t):
                if full0 is not None:
                    assert bool((outs[r][:, S.tolist()] == full0).all())
            del outs


@pytest.mark.parametrize("Nd", [1, 8, 64, 128])
@pytest.mark.parametrize("li", [0, 1])
def test_fwd_7b_decode(caat, Nd, li):
    w = ci.WORKLOADS["7b_prefill"]
    X, Wl, _ = ci.layer_tensors(w, li, N=Nd)
    S = caat.select_channels(w.h, w.p, 0)
    outs = caat.rowpar_linear_fwd(dev(X, "bf16"), _weight(Wl, "bf16", "nn"), w.t, sel_dev(S))
    torch().cuda.synchronize()
    want, _ = orc.rowpar_fwd(host_values(X, "bf16"), host_values(Wl, "bf16"), w.t, S)
    for r in range(w.t):
        check(to_f64(outs[r]), want[r], "bf16")


@pytest.fixture(params=["pair", "single"])
def bwd_cta(request, monkeypatch):
    """The backward GEMMs as CTA pairs (256 x 256 tiles, the default for
    256-column tiles above one 128-row block) or as single CTAs (CAAT_BWD_PAIR=0)."""
    monkeypatch.setenv("CAAT_BWD_PAIR", "1" if request.param == "pair" else "0")
    return request.param


# shapes whose backward tiles are 256 columns wide (CTA pairs by default):
# k_t = 256 with ragged rows (N = 300: the second pair's odd CTA reads only
# zero fill) and ragged channels (h = 264), k_t = 480 (two tiles, the last one
# 224 columns), and the most ranks the tensor-core backward takes (t = 16)
BWD_PAIR_SHAPES = [(2, 300, 256, 264), (4, 512, 480, 768), (16, 256, 256, 512)]


@pytest.mark.parametrize("t,N,kt,h", TC_SHAPES + BWD_PAIR_SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_bwd_tc_parity(caat, t, N, kt, h, mode, bwd_cta):
    for p in (0.0, 1.0 / h, 0.5, 0.75, 1.0 - 1.0 / h, 1.0):
        gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, p, 1, "bf16", mode, "nn", seed=3 * t + h)
        assert caat.last_kernel() == "rowpar_bwd_dw_tc"
        check(gX, wX, "bf16", bwd=True, what=("dX", p))
        check(gW, wW, "bf16", bwd=True, what=("dW", p))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("sel_kind", ["random", "contiguous_list", "contiguous_size"])
def test_bwd_token_split_parity(caat, mode, sel_kind, bwd_cta):
    """dW split over tokens: fp32 reduce-adds of the parts into the workspace's
    accumulator, then one rounding.  N = 2048 tokens are 32 k-blocks, which the
    split cuts into parts; k_t = 256 makes the column tiles 256 wide, so the
    default runs both GEMMs on CTA pairs; h = 520 leaves a pair whose odd CTA reads
    only zero fill.  S as a random index list, the contiguous S as a list, and the
    contiguous S by its size (the sum of the S channels formed once)."""
    T = torch()
    t, N, kt, h = 4, 2048, 256, 520
    K = kt * t
    X = ci.normal(1901, (N, K))
    Wl = ci.normal(1902, (K, h), std=0.02)
    G = ci.normal(1903, (t, N, h))
    if sel_kind == "contiguous_size":
        S = np.arange(256, dtype=np.int32)   # |S| a multiple of 64: the sum formed once
        sel = 256
    else:
        layout = caat.CAAT_S_RANDOM if sel_kind == "random" else caat.CAAT_S_CONTIGUOUS
        S = caat.select_channels(h, 0.5, layout, 1904)
        sel = sel_dev(S)
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Gd = [dev(G[r], "bf16") for r in range(t)]
    dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, sel, mode)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert caat.last_kernel() == "rowpar_bwd_dw_tc"
    wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                            np.stack([host_values(G[r], "bf16") for r in range(t)]), t, S, mode)
    check(to_f64(dX), wX, "bf16", bwd=True, what="dX")
    check(to_f64(dW), wW, "bf16", bwd=True, what="dW")


BWD_FULL = ([("130m", li, 0, 0.5, lay) for li in (0, 1) for lay in (0, 1)]
            + [("1.1b", li, 0, p, lay) for li in (0, 1) for p in (0.0, 0.25, 0.5, 0.75, 1.0)
               for lay in (0, 1)]
            + [(wn, li, 1, 0.5, 0) for wn in ("130m", "1.1b") for li in (0, 1)])


@pytest.mark.parametrize("wname,li,mode,p,layout", BWD_FULL)
def test_bwd_full_size_sampled(caat, wname, li, mode, p, layout):
    """Full workload sizes in the benchmark's launch configuration: dX on one
    sampled token row of every 128-row block (a row of dX needs only that row of
    the gradient), dW on one sampled channel of every 128-channel block (a column
    of dW needs only that channel of W and of the gradient, and whether it is in
    S), each over its whole other dimension.  The reduce placement runs the five
    p values at the 1.1B shapes; the other placement does not depend on S."""
    T = torch()
    w = ci.WORKLOADS[wname]
    X, Wl, G = ci.layer_tensors(w, li)
    S = caat.select_channels(w.h, p, layout, w.seeds()["perm"])
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Gd = [dev(G[r], "bf16") for r in range(w.t)]
    dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, w.t, _bench_sel(S, layout), mode)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert caat.last_kernel() == "rowpar_bwd_dw_tc"
    Xv, Wv = host_values(X, "bf16"), host_values(Wl, "bf16")
    Gv = np.stack([host_values(G[r], "bf16") for r in range(w.t)])
    rows = _block_samples(w.N, 128, 5 + li)
    wX, _ = orc.rowpar_bwd(Xv[rows], Wv, Gv[:, rows, :], w.t, S, mode)
    check(to_f64(dX[rows.tolist()]), wX, "bf16", bwd=True, what="dX")
    cols = _block_samples(w.h, 128, 7 + li)
    S_sub = np.nonzero(np.isin(cols, S))[0].astype(np.int32)
    _, wW = orc.rowpar_bwd(Xv, Wv[:, cols], Gv[:, :, cols], w.t, S_sub, mode)
    check(to_f64(dW[:, cols.tolist()]), wW, "bf16", bwd=True, what="dW")


@pytest.mark.parametrize("mode", [0, 1])
def test_bwd_tc_required_workspace_only(caat, mode):
    """A workspace with only the reduced-gradient region (no fp32 dW accumulator)
    takes the path without the token split; both paths match the oracle."""
    T = torch()
    t, N, kt, h = 8, 1024, 96, 768
    X = ci.normal(1201, (N, kt * t))
    Wl = ci.normal(1202, (kt * t, h), std=0.02)
    G = ci.normal(1203, (t, N, h))
    S = caat.select_channels(h, 0.5, 1, 9)
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Gd = [dev(G[r], "bf16") for r in range(t)]
    wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                            np.stack([host_values(G[r], "bf16") for r in range(t)]), t, S, mode)
    need = t * ((N * h * 2 + 255) // 256 * 256) if mode == 0 else 0
    full = caat.rowpar_linear_bwd_workspace(t, N, kt * t, h, 1, mode)
    assert full == need + (kt * t * h * 4 + 255) // 256 * 256
    for ws_bytes in (need, full):
        ws = T.empty(max(ws_bytes, 256), dtype=T.uint8, device="cuda") if ws_bytes else None
        dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, sel_dev(S), mode, workspace=ws)
        T.cuda.synchronize()
        assert caat.device_status() == 0
        check(to_f64(dX), wX, "bf16", bwd=True, what=ws_bytes)
        check(to_f64(dW), wW, "bf16", bwd=True, what=ws_bytes)


@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("N", [1, 3, 8, 9, 15])
def test_fwd_decode_parity(caat, t, N, monkeypatch):
    """Few tokens: the weight-streaming decode kernel (CUDA cores; the
    swapped-operand tensor-core kernel switched off)."""
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")
    h = 1000 if t != 16 else 520
    kt = 96 if t <= 8 else 64
    for p in (0.0, 0.5, 1.0):
        for layout in (0, 1):
            got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, layout, "bf16", "nn", seed=11 * t + N)
            assert caat.last_kernel() == "rowpar_fwd_decode"
            for r in range(t):
                check(got[r], want[r], "bf16", what=(r, p, layout), spread=spread)
            for r in range(1, t):
                assert np.array_equal(got[r][:, S], got[0][:, S])


@pytest.mark.parametrize("N", [16, 64, 100])
def test_fwd_small_n_tensor_core(caat, N, monkeypatch):
    """16 <= N < 128: the tile kernel with a partly empty 128-row tile (the
    swapped-operand kernel switched off)."""
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")
    t, kt, h = 8, 128, 512
    for layout in (0, 1):
        got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, 0.5, layout, "bf16", "nn", seed=N)
        assert caat.last_kernel() in ("rowpar_fwd_tc", "rowpar_fwd_decode")
        for r in range(t):
            check(got[r], want[r], "bf16", what=(r, layout), spread=spread)


@pytest.mark.parametrize("N,kt", [(1, 96), (8, 96), (300, 64), (2048, 96)])
def test_fwd_contiguous_null_sel_matches_index_list(caat, N, kt):
    """sel given as an int n (null pointer: S = first n channels) against the
    explicit index list of the same S, on every forward kernel.  The channels
    outside S are each rank's own partial, computed alike: the same bits.  On the
    tile kernel an index list with 0 < |S| < h sums the S channels from the ranks'
    rounded partials, the size form in fp32 over all of K: there both must match
    the oracle; the few-token kernels sum in fp32 either way: the same bits."""
    T = torch()
    t, h = 8, 768
    X = ci.normal(1301, (N, kt * t))
    Wl = ci.normal(1302, (kt * t, h), std=0.02)
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Xv, Wv = host_values(X, "bf16"), host_values(Wl, "bf16")
    for s in (0, 100, 384, 768):
        S = np.arange(s, dtype=np.int32)
        a = caat.rowpar_linear_fwd(Xd, Wd, t, sel_dev(S))
        ka = caat.last_kernel()
        b = caat.rowpar_linear_fwd(Xd, Wd, t, s)
        assert caat.last_kernel() == ka
        T.cuda.synchronize()
        for r in range(t):
            assert bool((a[r][:, s:].view(T.int16) == b[r][:, s:].view(T.int16)).all()), (s, r)
        if ka != "rowpar_fwd_tc" or s in (0, h):
            for r in range(t):
                assert bool((a[r].view(T.int16) == b[r].view(T.int16)).all()), (s, r)
        else:
            want, _ = orc.rowpar_fwd(Xv, Wv, t, S)
            parts, _ = orc.rowpar_fwd(Xv, Wv, t, np.zeros(0, np.int32))
            spread = np.zeros((N, h))
            spread[:, :s] = np.abs(parts).sum(axis=0)[:, :s]
            for r in range(t):
                check(to_f64(a[r]), want[r], "bf16", spread=spread, what=("list", s, r))
                check(to_f64(b[r]), want[r], "bf16", what=("size", s, r))
                assert bool((a[r][:, :s] == a[0][:, :s]).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pcr_contiguous_null_sel_bitexact(caat, dtype):
    t, N, h = 8, 257, 768
    Y = ci.normal(1401, (t, N, h))
    from tests.gpu_helpers import words
    for s in (0, 5, 384, 768):
        ins = [dev(Y[r], dtype) for r in range(t)]
        outs = caat.partial_channel_reduce(ins, s)
        torch().cuda.synchronize()
        got = np.stack([words(o) for o in outs])
        if dtype == "f32":
            want = orc.pcr_f32(Y, np.arange(s))[0].view(np.uint32)
        else:
            want = orc.pcr_bf16(ci.bf16_words(Y), np.arange(s))[0]
        np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("s", [0, 64, 384, 448, 768, 100])
@pytest.mark.parametrize("kt", [96, 256, 384])
def test_bwd_contiguous_reduce_once(caat, s, kt, bwd_cta):
    """Contiguous S given as an int: with |S| a multiple of 64 the backward reduces
    only the S channels once (the GEMMs read the other channels straight from each
    rank's gradient); other sizes take the materialising path.  Both match the
    oracle."""
    T = torch()
    t, N, h = 8, 1024, 768
    X = ci.normal(1501 + kt, (N, kt * t))
    Wl = ci.normal(1502 + kt, (kt * t, h), std=0.02)
    G = ci.normal(1503 + kt, (t, N, h))
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Gd = [dev(G[r], "bf16") for r in range(t)]
    dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, s, caat.CAAT_BWD_REDUCE_DOUT)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert caat.last_kernel() == "rowpar_bwd_dw_tc"
    wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                            np.stack([host_values(G[r], "bf16") for r in range(t)]), t,
                            np.arange(s), 0)
    check(to_f64(dX), wX, "bf16", bwd=True)
    check(to_f64(dW), wW, "bf16", bwd=True)


@pytest.mark.parametrize("s", [64, 2048, 3072, 4096])
def test_bwd_contiguous_reduce_once_wide(caat, s):
    """The reduce-once path at h = 4096: S from 64 channels (8 chunks of 8 per row, many
    rows per block) to 4096 (512 chunks per row, two blocks across a row), ragged
    token count."""
    T = torch()
    t, N, kt, h = 4, 200, 64, 4096
    X = ci.normal(1701, (N, kt * t))
    Wl = ci.normal(1702, (kt * t, h), std=0.02)
    G = ci.normal(1703, (t, N, h))
    Xd, Wd = dev(X, "bf16"), _weight(Wl, "bf16", "nn")
    Gd = [dev(G[r], "bf16") for r in range(t)]
    dX, dW = caat.rowpar_linear_bwd(Xd, Wd, Gd, t, s, caat.CAAT_BWD_REDUCE_DOUT)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    assert caat.last_kernel() == "rowpar_bwd_dw_tc"
    wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                            np.stack([host_values(G[r], "bf16") for r in range(t)]), t,
                            np.arange(s), 0)
    check(to_f64(dX), wX, "bf16", bwd=True)
    check(to_f64(dW), wW, "bf16", bwd=True)


@pytest.mark.parametrize("t", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("N", [1, 3, 8, 15, 16, 17, 33, 48, 64, 65, 100, 128])
def test_fwd_skinny_parity(caat, t, N):
    """Few tokens (N <= 128, t <= 8): the swapped-operand tensor-core kernel, one
    cluster of t shard-CTAs per 128-channel block; ragged channel blocks (h = 1000)
    and ragged shards (k_t = 136: the last 64-wide k block is part zero fill).
    t = 3, 5, 7 give the CTAs channel slices of the S sum (128 / t channels)
    that are neither equal nor multiples of the 8-channel store."""
    for h, kt in ((1000, 136), (512, 64)):
        for p in (0.0, 0.5, 1.0):
            for layout in (0, 1):
                got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, layout, "bf16", "nn", seed=13 * t + N + h)
                assert caat.last_kernel() == "rowpar_fwd_skinny_tc"
                for r in range(t):
                    check(got[r], want[r], "bf16", what=(h, r, p, layout), spread=spread)
                for r in range(1, t):
                    assert np.array_equal(got[r][:, S], got[0][:, S])


@pytest.mark.parametrize("t", [1, 3, 8])
@pytest.mark.parametrize("N", [129, 200, 256, 385])
def test_fwd_skinny_token_chunks(caat, t, N, monkeypatch):
    """Above 128 tokens the swapped-operand kernel runs one cluster per
    (128-channel block, chunk of 128 tokens), taken here by raising its token
    bound: every chunk's rows land in their own output rows, the last chunk
    ragged (N = 129 leaves one row in it), and the S sums agree across ranks."""
    monkeypatch.setenv("CAAT_FWD_SKINNY_MAX", "8192")
    for h, kt in ((1000, 136), (512, 64)):
        for p, layout in ((0.5, 0), (0.5, 1), (1.0, 0)):
            got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, layout, "bf16", "nn", seed=7 * t + N + h)
            assert caat.last_kernel() == "rowpar_fwd_skinny_tc"
            for r in range(t):
                check(got[r], want[r], "bf16", what=(h, r, p, layout), spread=spread)
            for r in range(1, t):
                assert np.array_equal(got[r][:, S], got[0][:, S])


def test_fwd_skinny_token_chunks_guard(caat, monkeypatch):
    # token chunks into rank outputs with a row stride wider than h: the padding
    # columns and the row after the last stay untouched
    monkeypatch.setenv("CAAT_FWD_SKINNY_MAX", "8192")
    T = torch()
    t, N, kt, h, ld = 4, 300, 64, 200, 264
    X = ci.normal(907, (N, kt * t))
    Wl = ci.normal(908, (kt * t, h), std=0.02)
    S = caat.select_channels(h, 0.5, 1, 6)
    bufs = [T.full((N + 1, ld), 7.0, dtype=T.bfloat16, device="cuda") for _ in range(t)]
    outs = [b[:N, :h] for b in bufs]
    caat.rowpar_linear_fwd(dev(X, "bf16"), _weight(Wl, "bf16", "nn"), t, sel_dev(S), outs=outs)
    T.cuda.synchronize()
    assert caat.last_kernel() == "rowpar_fwd_skinny_tc"
    for b in bufs:
        assert bool((b[:, h:] == 7.0).all()) and bool((b[N] == 7.0).all())
    want, _ = orc.rowpar_fwd(host_values(X, "bf16"), host_values(Wl, "bf16"), t, S)
    for r in range(t):
        check(to_f64(outs[r]), want[r], "bf16")


def test_fwd_skinny_declines_to_other_kernels(caat):
    """Shapes the swapped-operand kernel does not take still run: t = 16 (above
    the portable cluster size) and k_t < 64 go to the CUDA-core decode kernel."""
    for t, kt in ((16, 64), (8, 32)):
        got, want, _, spread = _fwd_case(caat, t, 4, kt * t, 256, 0.5, 1, "bf16", "nn", seed=t + kt)
        assert caat.last_kernel() == "rowpar_fwd_decode"
        for r in range(t):
            check(got[r], want[r], "bf16", spread=spread)


@pytest.mark.parametrize("N", [5, 40, 100])
def test_fwd_skinny_output_guard(caat, N):
    # rank outputs with a row stride wider than h and a ragged last channel block
    # (h = 200): the padding columns must stay untouched
    T = torch()
    t, kt, h, ld = 4, 64, 200, 264
    X = ci.normal(905, (N, kt * t))
    Wl = ci.normal(906, (kt * t, h), std=0.02)
    S = caat.select_channels(h, 0.5, 1, 6)
    bufs = [T.full((N + 1, ld), 7.0, dtype=T.bfloat16, device="cuda") for _ in range(t)]
    outs = [b[:N, :h] for b in bufs]
    caat.rowpar_linear_fwd(dev(X, "bf16"), _weight(Wl, "bf16", "nn"), t, sel_dev(S), outs=outs)
    T.cuda.synchronize()
    assert caat.last_kernel() == "rowpar_fwd_skinny_tc"
    for b in bufs:
        assert bool((b[:, h:] == 7.0).all()) and bool((b[N] == 7.0).all())
    want, _ = orc.rowpar_fwd(host_values(X, "bf16"), host_values(Wl, "bf16"), t, S)
    for r in range(t):
        check(to_f64(outs[r]), want[r], "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t,N,kt,h", [(64, 9, 2, 24), (64, 130, 4, 40), (32, 3, 8, 16)])
def test_layer_maximum_rank_count(caat, dtype, t, N, kt, h):
    """t up to 64: forward and both backward placements on the kernels that take it."""
    for p in (0.0, 0.5, 1.0):
        got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, 1, dtype, "nn", seed=t + N)
        for r in range(t):
            check(got[r], want[r], dtype, what=("fwd", r, p), spread=spread)
        for r in range(1, t):
            assert np.array_equal(got[r][:, S], got[0][:, S])
        for mode in (0, 1):
            gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, p, 1, dtype, mode, "nn", seed=t + N)
            check(gX, wX, dtype, bwd=True, what=("dX", mode, p))
            check(gW, wW, dtype, bwd=True, what=("dW", mode, p))


@pytest.mark.parametrize("t", [16, 17])
def test_layer_tensor_core_rank_limit(caat, t):
    """t = 16 is the largest rank count of the tile kernels (one output tensor map
    per rank); t = 17 falls back to the CUDA-core kernels.  Both match the oracle."""
    N, kt, h = 256, 64, 256
    got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, 0.5, 1, "bf16", "nn", seed=t)
    assert caat.last_kernel() == ("rowpar_fwd_tc" if t <= 16 else "rowpar_fwd_simt")
    for r in range(t):
        check(got[r], want[r], "bf16", spread=spread)
    gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, 0.5, 1, "bf16", 0, "nn", seed=t)
    check(gX, wX, "bf16", bwd=True)
    check(gW, wW, "bf16", bwd=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t,N,kt,h", [(2, 1, 1, 1), (3, 4, 1, 2), (1, 1, 1, 1), (4, 17, 1, 5)])
def test_layer_degenerate_shapes(caat, dtype, t, N, kt, h):
    """One channel, one token, one element per shard."""
    for p in (0.0, 1.0):
        got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, p, 0, dtype, "rm", seed=t + h)
        for r in range(t):
            check(got[r], want[r], dtype, spread=spread)
        gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, p, 0, dtype, 0, "rm", seed=t + h)
        check(gX, wX, dtype, bwd=True)
        check(gW, wW, dtype, bwd=True)


@pytest.mark.parametrize("layout", [0, 1])
def test_fwd_bwd_largest_h(caat, layout, fwd_mode):
    """The largest channel count the tensor-core forward takes (h = 32768: a
    1024-word S bitmap, 128 channel blocks of 256 -- h is no multiple of 192, so
    the 192-wide modes run 256-wide tiles), random and contiguous S, in every
    forward mode; and the backward in both placements."""
    t, N, kt, h = 2, 256, 64, 32768
    got, want, S, spread = _fwd_case(caat, t, N, kt * t, h, 0.5, layout, "bf16", "nn", seed=31)
    assert caat.last_kernel() == "rowpar_fwd_tc"
    for r in range(t):
        check(got[r], want[r], "bf16", what=r, spread=spread)
    if fwd_mode != "2":
        return                      # the backward does not depend on the forward mode
    for mode in (0, 1):
        gX, gW, wX, wW = _bwd_case(caat, t, N, kt * t, h, 0.5, layout, "bf16", mode, seed=32)
        check(gX, wX, "bf16", bwd=True, what=("dX", mode))
        check(gW, wW, "bf16", bwd=True, what=("dW", mode))
