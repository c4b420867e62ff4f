"""Host-side checks of the C ABI (no GPU): the library builds, loads, exports
every function ``include/caat.h`` declares, builds S bit-exactly like the oracle,
and rejects invalid arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from partial_activation_sync_gb300 import build
    build.build()
    from partial_activation_sync_gb300 import _lib
    return _lib.load()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(caat_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert "caat_partial_channel_reduce" in declared
    assert "caat_rowpar_linear_fwd" in declared
    assert "caat_rowpar_linear_bwd" in declared
    assert "caat_select_channels" in declared
    for name in declared:
        assert hasattr(lib, name), name
    from partial_activation_sync_gb300 import _lib
    assert set(_lib.EXPORTS) <= declared


def test_built_for_sm103a():
    from partial_activation_sync_gb300 import build
    assert ["-gencode", "arch=compute_103a,code=sm_103a"] == build.ARCH


@pytest.mark.parametrize("h", [0, 1, 7, 12, 768, 2048, 4096, 5000])
def test_select_channels_matches_oracle(lib, h):
    import partial_activation_sync_gb300 as caat
    for layout in (0, 1):
        for p in (0.0, 0.25, 0.5, 0.75, 1.0, 0.3333):
            for seed in (0, 4003, 2**63 + 5):
                a = caat.select_channels(h, p, layout, seed)
                b = orc.select_channels(h, p, layout, seed)
                np.testing.assert_array_equal(a, b)


def test_select_channels_rejects_bad_args(lib):
    n = ctypes.c_int64(0)
    idx = (ctypes.c_int32 * 8)()
    assert lib.caat_select_channels(8, 1.5, 0, 0, idx, ctypes.byref(n)) == 1
    assert lib.caat_select_channels(8, float("nan"), 0, 0, idx, ctypes.byref(n)) == 1
    assert lib.caat_select_channels(8, 0.5, 7, 0, idx, ctypes.byref(n)) == 1
    assert lib.caat_select_channels(-1, 0.5, 0, 0, idx, ctypes.byref(n)) == 1
    assert lib.caat_select_channels(8, 0.5, 0, 0, None, ctypes.byref(n)) == 1
    assert lib.caat_select_channels(8, 0.5, 0, 0, idx, None) == 1
    assert lib.caat_select_channels(0, 0.5, 0, 0, None, ctypes.byref(n)) == 0 and n.value == 0


def _ptrs(vals):
    from partial_activation_sync_gb300 import _lib
    return _lib.ptr_array(vals)


def test_pcr_rejects_bad_args_without_launch(lib):
    # fake, never dereferenced device addresses: every call must fail validation
    a, b, c = 1 << 20, 2 << 20, 3 << 20
    sel = ctypes.c_void_p(4 << 20)
    f = lib.caat_partial_channel_reduce
    assert f(0, 4, 8, 0, _ptrs([a]), 8, _ptrs([b]), 8, sel, 2, None) == 1        # t < 1
    assert f(65, 4, 8, 0, _ptrs([a]), 8, _ptrs([b]), 8, sel, 2, None) == 1       # t > 64
    assert f(1, 4, 8, 5, _ptrs([a]), 8, _ptrs([b]), 8, sel, 2, None) == 1        # dtype
    assert f(1, 4, 8, 0, _ptrs([a]), 7, _ptrs([b]), 8, sel, 2, None) == 1        # ld_in < h
    assert f(1, 4, 8, 0, _ptrs([a]), 8, _ptrs([b]), 8, sel, 9, None) == 1        # n_sel > h
    assert f(1, 4, 8, 0, _ptrs([a]), 8, _ptrs([b]), 8, None, -1, None) == 1      # n_sel < 0
    assert f(2, 4, 8, 0, _ptrs([a, b]), 8, _ptrs([a, c]), 8, sel, 2, None) == 1  # half in place
    assert f(2, 4, 8, 0, _ptrs([a, b]), 8, _ptrs([c, c]), 8, sel, 2, None) == 1  # outputs overlap
    assert f(2, 4, 8, 0, _ptrs([a, b]), 8, _ptrs([b + 16, c]), 8, sel, 2, None) == 1  # out hits in
    assert f(2, 4, 8, 0, _ptrs([a, 0]), 8, _ptrs([b, c]), 8, sel, 2, None) == 1  # null pointer
    assert f(2, 4, 8, 0, _ptrs([a, b]), 8, _ptrs([a, b]), 16, sel, 2, None) == 1  # in place, ld differ
    assert f(2, 4, 8, 0, _ptrs([a, b]), 8, _ptrs([c, (4 << 20) - 8]), 8, sel, 2, None) == 1  # out hits sel


def test_layer_rejects_bad_args_without_launch(lib):
    X, W, Y0, Y1 = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    sel = ctypes.c_void_p(5 << 20)
    f = lib.caat_rowpar_linear_fwd
    # K % t != 0
    assert f(2, 4, 7, 8, 1, X, 7, W, 1, 7, _ptrs([Y0, Y1]), 8, sel, 2, None) == 1
    # ldx < K
    assert f(2, 4, 8, 8, 1, X, 4, W, 1, 8, _ptrs([Y0, Y1]), 8, sel, 2, None) == 1
    # W strides that alias elements
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 1, _ptrs([Y0, Y1]), 8, sel, 2, None) == 1
    # ldy < h
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 4, sel, 2, None) == 1
    # outputs overlap
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y0]), 8, sel, 2, None) == 1
    # n_sel > h
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, sel, 9, None) == 1
    # an output overlaps W (column-major [8, 8] bf16: 128 bytes from W) or the index list
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, W + 64]), 8, sel, 2, None) == 1
    assert f(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, (5 << 20) - 16]), 8, sel, 2, None) == 1
    g = lib.caat_rowpar_linear_bwd
    f_ws = lib.caat_rowpar_linear_bwd_workspace
    # two [4, 8] bf16 buffers (256-byte rounded) + fp32 dW accumulator [8, 8] (256 bytes)
    assert f_ws(2, 4, 8, 8, 1, 0) == 2 * 256 + 256
    assert f_ws(2, 4, 8, 8, 1, 1) == 256            # no reduced gradient without the reduce
    assert f_ws(2, 4, 8, 8, 0, 0) == 2 * 256        # fp32: no accumulator
    assert f_ws(2, 4, 8, 8, 0, 1) == 0
    # workspace missing for the reduce-dOut mode
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, 6 << 20, 8, 7 << 20, 1, 8,
             sel, 2, 0, None, 0, None) == 1
    # bad mode
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, 6 << 20, 8, 7 << 20, 1, 8,
             sel, 2, 9, None, 0, None) == 1
    # written regions that overlap an input or each other (mode NO_REDUCE: no workspace
    # needed, so only the overlap can fail the call)
    dX, dW = 6 << 20, 7 << 20
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, Y1 + 32, 8, dW, 1, 8,
             sel, 2, 1, None, 0, None) == 1                       # dX over a gradient
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, dX, 8, X + 16, 1, 8,
             sel, 2, 1, None, 0, None) == 1                       # dW over X
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, dX, 8, W, 1, 8,
             sel, 2, 1, None, 0, None) == 1                       # dW over W
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, dX, 8, dX + 32, 1, 8,
             sel, 2, 1, None, 0, None) == 1                       # dX and dW overlap
    # the used workspace (256-byte aligned) over dX, and over a gradient
    ws = 8 << 20
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, Y1]), 8, ws + 64, 8, dW, 1, 8,
             sel, 2, 0, ws, 768, None) == 1
    assert g(2, 4, 8, 8, 1, X, 8, W, 1, 8, _ptrs([Y0, ws + 256]), 8, dX, 8, dW, 1, 8,
             sel, 2, 0, ws, 768, None) == 1


def test_compact_layer_rejects_bad_args_without_launch(lib):
    # compact outputs: YS [4, n_sel] and YN[r] [4, 8 - n_sel]; fake device pointers,
    # every case returns before anything touches the device
    X, W, YS, Y0, Y1 = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20
    sel, ws = ctypes.c_void_p(9 << 20), 10 << 20
    f = lib.caat_rowpar_linear_fwd_compact
    ok = [2, 4, 8, 8, 1, X, 8, W, 1, 8, YS, 2, _ptrs([Y0, Y1]), 6, None, 2, None, 0, None]

    def fc(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert fc() == 2                                      # n_sel % 64
    assert fc(a4=0) == 2                                  # fp32
    assert fc(a11=1) == 1                                 # ldys < n_sel
    assert fc(a13=5) == 1                                 # ldyn < h - n_sel
    assert fc(a10=None) == 1                              # no YS
    assert fc(a12=_ptrs([Y0, YS + 8])) == 1               # YN over YS
    assert fc(a12=_ptrs([Y0, Y0 + 4])) == 1               # YN overlap
    assert fc(a10=X + 2) == 1                             # YS over X
    assert fc(a15=9) == 1                                 # n_sel > h
    assert fc(a14=sel) == 1                               # an index list needs the permuted W
    assert fc(a14=sel, a16=ws, a17=64) == 1               # ... of h*K*2 = 128 bytes (256 rounded)
    assert fc(a14=sel, a16=ws + 16, a17=256) == 1         # ... 256-byte aligned
    assert fc(a14=sel, a16=YS, a17=256) == 1              # ... not over an output
    assert fc(a14=sel, a16=ws, a17=256) == 2              # valid, but n_sel % 64
    g = lib.caat_rowpar_linear_bwd_compact
    dX, dW = 6 << 20, 7 << 20
    okb = [2, 4, 8, 8, 1, X, 8, W, 1, 8, YS, 2, _ptrs([Y0, Y1]), 6, dX, 8, dW, 1, 8, None, 2, None, 0, None]

    def gc(**kw):
        a = list(okb)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return g(*a)
    assert gc() == 2                                      # n_sel % 64
    assert gc(a11=1) == 1                                 # lddys < n_sel
    assert gc(a13=5) == 1                                 # lddyn < h - n_sel
    assert gc(a14=YS + 4) == 1                            # dX over dYS
    assert gc(a16=Y1 + 8) == 1                            # dW over a dYN
    assert gc(a16=dX + 16) == 1                           # dX and dW overlap
    assert gc(a12=None) == 1                              # no dYN
    assert gc(a19=sel) == 1                               # index list: W copy + dW staging required
    assert gc(a19=sel, a21=ws, a22=256) == 1              # 256 + 256 bytes needed
    assert gc(a19=sel, a21=ws, a22=512) == 2              # valid, but n_sel % 64
    w = lib.caat_rowpar_linear_compact_workspace
    assert w(2, 4, 8, 8, 1, 0, 0) == 0
    assert w(2, 4, 8, 8, 1, 1, 0) == 256                  # W [8, 8] bf16, rounded up
    assert w(2, 4, 8, 8, 1, 0, 1) == 256                  # fp32 accumulator [8, 8]
    assert w(2, 4, 8, 8, 1, 1, 1) == 768                  # W, dW staging, accumulator
    assert w(0, 4, 8, 8, 1, 1, 1) == 0


def test_colpar_rejects_bad_args_without_launch(lib):
    A0, A1, W1, Z = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    sel = ctypes.c_void_p(5 << 20)
    f = lib.caat_colpar_linear_fwd
    # K % t != 0
    assert f(2, 4, 8, 7, 1, _ptrs([A0, A1]), 8, W1, 7, 1, Z, 7, None) == 1
    # lda < h
    assert f(2, 4, 8, 8, 1, _ptrs([A0, A1]), 4, W1, 8, 1, Z, 8, None) == 1
    # ldz < K
    assert f(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, Z, 4, None) == 1
    # W1 strides that alias elements
    assert f(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 1, 1, Z, 8, None) == 1
    # Z overlaps an input
    assert f(2, 4, 8, 8, 1, _ptrs([A0, Z]), 8, W1, 8, 1, Z, 8, None) == 1
    # null input pointer
    assert f(2, 4, 8, 8, 1, _ptrs([A0, 0]), 8, W1, 8, 1, Z, 8, None) == 1
    # Z overlaps W1
    assert f(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, W1 + 32, 8, None) == 1
    g = lib.caat_colpar_linear_bwd
    dZ, dA0, dA1, dW1 = 6 << 20, 7 << 20, 8 << 20, 9 << 20
    # optional fp32 accumulator of dW1 [8, 8]: 256 bytes; none for fp32
    assert lib.caat_colpar_linear_bwd_workspace(2, 4, 8, 8, 1) == 256
    assert lib.caat_colpar_linear_bwd_workspace(2, 4, 8, 8, 0) == 0
    # dA outputs overlap each other
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA0]), 8,
             dW1, 8, 1, sel, 2, None, 0, None) == 1
    # dA overlaps an input
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, A1]), 8,
             dW1, 8, 1, sel, 2, None, 0, None) == 1
    # n_sel > h
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             dW1, 8, 1, sel, 9, None, 0, None) == 1
    # dW1 strides that alias elements
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             dW1, 1, 1, sel, 2, None, 0, None) == 1
    # ldda < h
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 4,
             dW1, 8, 1, sel, 2, None, 0, None) == 1
    # dA overlaps W1; dW1 overlaps dZ, an input block or an output block
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, W1 + 16]), 8,
             dW1, 8, 1, sel, 2, None, 0, None) == 1
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             dZ + 16, 8, 1, sel, 2, None, 0, None) == 1
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             A1, 8, 1, sel, 2, None, 0, None) == 1
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             dA1 + 8, 8, 1, sel, 2, None, 0, None) == 1
    # the fp32 accumulator (256-byte aligned workspace) over dZ
    assert g(2, 4, 8, 8, 1, _ptrs([A0, A1]), 8, W1, 8, 1, dZ, 8, _ptrs([dA0, dA1]), 8,
             dW1, 8, 1, sel, 2, dZ, 256, None) == 1


def test_status_strings(lib):
    for code in range(5):
        assert lib.caat_status_string(code).startswith(b"CAAT_")
    assert lib.caat_status_string(99) == b"CAAT: unknown status"


def test_debug_set_wait_validates(lib):
    """The failure-path test hook rejects limits outside 1 us .. 10 s and unknown
    injections, and accepts the reset (0, none); it launches nothing."""
    assert lib.caat_debug_set_wait(999, 0) == 1
    assert lib.caat_debug_set_wait(10_000_000_001, 0) == 1
    assert lib.caat_debug_set_wait(1_000_000, 7) == 1
    assert lib.caat_debug_set_wait(1_000_000, 1) == 0
    assert lib.caat_debug_set_wait(0, 0) == 0


def test_exchange_steps_reject_bad_args_without_launch(lib):
    """pack / unpack / fold: sizes, leading dimensions, null data pointers and
    overlapping buffers are rejected before any launch (fake device addresses)."""
    vp = ctypes.c_void_p
    Y, P = vp(0x100000), vp(0x900000)
    # pack: n_sel > h, ld below the row, null P, P overlapping Y
    assert lib.caat_pcr_pack(4, 8, 1, Y, 8, None, 9, P, 9, None) == 1
    assert lib.caat_pcr_pack(4, 8, 1, Y, 7, None, 4, P, 4, None) == 1
    assert lib.caat_pcr_pack(4, 8, 1, Y, 8, None, 4, None, 4, None) == 1
    assert lib.caat_pcr_pack(4, 8, 1, Y, 8, None, 4, vp(0x100000 + 8), 4, None) == 1
    assert lib.caat_pcr_pack(0, 8, 1, Y, 8, None, 4, P, 4, None) == 0          # nothing to move
    # unpack: no outputs, too many, overlapping outputs, output overlapping P
    arr = (ctypes.c_void_p * 2)(0x100000, 0x100000 + 16)
    assert lib.caat_pcr_unpack(4, 8, 1, P, 4, None, 4, arr, 0, 8, None) == 1
    assert lib.caat_pcr_unpack(4, 8, 1, P, 4, None, 4, arr, 65, 8, None) == 1
    assert lib.caat_pcr_unpack(4, 8, 1, P, 4, None, 4, arr, 2, 8, None) == 1
    one = (ctypes.c_void_p * 1)(0x900000 + 4)
    assert lib.caat_pcr_unpack(4, 8, 1, P, 4, None, 4, one, 1, 8, None) == 1
    # fold: t out of range, blocks overlapping each other, output inside the input
    assert lib.caat_rank_fold(0, 4, 8, 1, Y, 8, 32, P, 8, None) == 1
    assert lib.caat_rank_fold(2, 4, 8, 1, Y, 8, 16, P, 8, None) == 1
    assert lib.caat_rank_fold(2, 4, 8, 1, Y, 8, 32, vp(0x100000 + 40), 8, None) == 1
    assert lib.caat_rank_fold(2, 0, 8, 1, Y, 8, 32, P, 8, None) == 0         # nothing to fold
