"""The backward entry point that allocates nothing (caat_rowpar_linear_bwd_noalloc).

Some callers cannot call cudaMalloc -- a framework that owns every byte of
device memory through its own pool, or a process with a memory budget fixed at
start-up -- so they cannot hand the regular backward a workspace.  This entry
point uses the library's own fixed-size scratch array instead.  Here it is
called straight through the C ABI and compared with the regular entry point
(which gets a workspace from PyTorch), twice in a row with different inputs, so
that a result left over in the shared array from the first call would show.

The file is named to be collected last."""
import ctypes

import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import TOL, check, dev, host_values, rel_fro, sel_dev, to_f64, torch

pytestmark = pytest.mark.gpu

MAX_BYTES = 16 << 20


def _fn():
    from partial_activation_sync_gb300 import _lib
    L = _lib.load()
    f = L.caat_rowpar_linear_bwd_noalloc
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.POINTER(ctypes.c_void_p), ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f, _lib


def _call_noalloc(f, _lib, t, X, Wst, G, dX, dWst, sel, mode):
    """sel: a device int32 tensor of S, or an int s for the contiguous S = the
    first s channels (passed as a null index pointer)."""
    T = torch()
    sp, ns = (None, int(sel)) if isinstance(sel, int) else (sel.data_ptr(), sel.numel())
    N, K = X.shape
    h = Wst.shape[0]
    code = 1 if X.dtype == T.bfloat16 else 0
    stream = ctypes.c_void_p(T.cuda.current_stream().cuda_stream)
    # W and dW in the nn.Linear layout: logical [K, h] with strides (1, K)
    return f(t, N, K, h, code, X.data_ptr(), K, Wst.data_ptr(), 1, K,
             _lib.ptr_array([g.data_ptr() for g in G]), h, dX.data_ptr(), K,
             dWst.data_ptr(), 1, K, sp, ns, mode, stream)


@pytest.mark.parametrize("dtype,t,N,K,h", [("bf16", 8, 512, 3072, 768), ("f32", 4, 200, 256, 520)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, t, N, K, h):
    import partial_activation_sync_gb300 as caat
    T = torch()
    f, _lib = _fn()
    assert t * N * h * (2 if dtype == "bf16" else 4) <= MAX_BYTES
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 123)
    sel = sel_dev(S)
    for call, seed in enumerate((1, 2)):
        X = ci.normal(50 + seed, (N, K))
        Wl = ci.normal(60 + seed, (K, h), std=0.02)
        G = ci.normal(70 + seed, (t, N, h))
        Xd = dev(X, dtype)
        Wst = dev(np.ascontiguousarray(Wl.T), dtype)
        Gd = [dev(G[r], dtype) for r in range(t)]
        dX_ref, dW_ref = caat.rowpar_linear_bwd(Xd, Wst.t(), Gd, t, sel, caat.CAAT_BWD_REDUCE_DOUT)
        dX = T.full((N, K), float("nan"), dtype=Xd.dtype, device="cuda")
        dWst = T.full((h, K), float("nan"), dtype=Xd.dtype, device="cuda")
        st = _call_noalloc(f, _lib, t, Xd, Wst, Gd, dX, dWst, sel, 0)
        assert st == 0, _lib.load().caat_status_string(st)
        T.cuda.synchronize()
        assert caat.device_status() == 0
        assert rel_fro(to_f64(dX), to_f64(dX_ref)) <= TOL[dtype], call
        assert rel_fro(to_f64(dWst.t()), to_f64(dW_ref)) <= TOL[dtype], call
        # and both against the oracle
        wX, wW = orc.rowpar_bwd(host_values(X, dtype), host_values(Wl, dtype),
                                np.stack([host_values(G[r], dtype) for r in range(t)]), t, S, 0)
        check(to_f64(dX), wX, dtype, bwd=True, what=("dX", call))
        check(to_f64(dWst.t()), wW, dtype, bwd=True, what=("dW", call))


# Shapes whose scratch also holds the fp32 dW accumulator, so the token-split dW
# reduction runs out of the shared array too:
#  - contiguous S given by its size (n_sel a multiple of 64): the sum of the S
#    channels [N, n_sel] sits at the start of the array and the accumulator after
#    the reduced-gradient region (8 x 512 x 768 x 2 B = 6 MiB + 768 x 768 x 4 B);
#  - the placement without the reduce: the accumulator alone, from offset 0.
@pytest.mark.parametrize("mode,sel_kind", [(0, "contiguous"), (1, "random"), (1, "contiguous")])
def test_noalloc_accumulator_paths_match_twice(mode, sel_kind):
    import partial_activation_sync_gb300 as caat
    T = torch()
    f, _lib = _fn()
    t, N, K, h = 8, 512, 768, 768
    need = t * N * h * 2 if mode == 0 else 0
    assert need + K * h * 4 <= MAX_BYTES
    if sel_kind == "contiguous":
        sel = h // 2
    else:
        sel = sel_dev(caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 321))
    for call, seed in enumerate((3, 4)):
        X = ci.normal(80 + seed, (N, K))
        Wl = ci.normal(90 + seed, (K, h), std=0.02)
        G = ci.normal(100 + seed, (t, N, h))
        Xd = dev(X, "bf16")
        Wst = dev(np.ascontiguousarray(Wl.T), "bf16")
        Gd = [dev(G[r], "bf16") for r in range(t)]
        dX_ref, dW_ref = caat.rowpar_linear_bwd(Xd, Wst.t(), Gd, t, sel, mode)
        dX = T.full((N, K), float("nan"), dtype=Xd.dtype, device="cuda")
        dWst = T.full((h, K), float("nan"), dtype=Xd.dtype, device="cuda")
        st = _call_noalloc(f, _lib, t, Xd, Wst, Gd, dX, dWst, sel, mode)
        assert st == 0, _lib.load().caat_status_string(st)
        T.cuda.synchronize()
        assert caat.device_status() == 0
        assert rel_fro(to_f64(dX), to_f64(dX_ref)) <= TOL["bf16"], call
        assert rel_fro(to_f64(dWst.t()), to_f64(dW_ref)) <= TOL["bf16"], call
        S = np.arange(sel, dtype=np.int32) if isinstance(sel, int) else sel.cpu().numpy()
        wX, wW = orc.rowpar_bwd(host_values(X, "bf16"), host_values(Wl, "bf16"),
                                np.stack([host_values(G[r], "bf16") for r in range(t)]), t, S, mode)
        check(to_f64(dX), wX, "bf16", bwd=True, what=("dX", call))
        check(to_f64(dWst.t()), wW, "bf16", bwd=True, what=("dW", call))


def test_noalloc_rejects_sizes_beyond_the_scratch():
    import partial_activation_sync_gb300 as caat
    T = torch()
    f, _lib = _fn()
    t, N, K, h = 8, 2048, 64, 1024          # 8 * 2048 * 1024 * 2 B = 32 MiB > 16 MiB
    X = T.zeros((N, K), dtype=T.bfloat16, device="cuda")
    Wst = T.zeros((h, K), dtype=T.bfloat16, device="cuda")
    G = [T.zeros((N, h), dtype=T.bfloat16, device="cuda") for _ in range(t)]
    dX = T.zeros((N, K), dtype=T.bfloat16, device="cuda")
    dWst = T.zeros((h, K), dtype=T.bfloat16, device="cuda")
    sel = sel_dev(np.arange(h // 2, dtype=np.int32))
    assert _call_noalloc(f, _lib, t, X, Wst, G, dX, dWst, sel, 0) == 1   # CAAT_ERR_INVALID_ARG
    # the same size without the reduce needs no scratch and runs; so does the
    # reduce with an empty S or with one rank (nothing to sum)
    assert _call_noalloc(f, _lib, t, X, Wst, G, dX, dWst, sel, 1) == 0
    assert _call_noalloc(f, _lib, t, X, Wst, G, dX, dWst, 0, 0) == 0
    Xw = T.zeros((N, t * K), dtype=T.bfloat16, device="cuda")
    Ww = T.zeros((h, t * K), dtype=T.bfloat16, device="cuda")
    dXw = T.zeros((N, t * K), dtype=T.bfloat16, device="cuda")
    dWw = T.zeros((h, t * K), dtype=T.bfloat16, device="cuda")
    assert _call_noalloc(f, _lib, 1, Xw, Ww, G[:1], dXw, dWw, sel, 0) == 0
    T.cuda.synchronize()
    assert caat.device_status() == 0
