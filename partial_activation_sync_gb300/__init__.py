"""GB300 (sm_103a) partial channel-reduce for tensor-parallel layers (CAAT-Net).

Thin PyTorch binding over the C ABI of ``include/caat.h``: every function below
only marshals tensors (device pointers, sizes, strides, the current CUDA stream)
into one library call; all arithmetic runs in the library's CUDA kernels.

"Tensor-Parallelism with Partially Synchronized Activations" (NeurIPS 2025),
Introduction: the partial channel-reduce sums only a subset S of the hidden
channels over the t tensor-parallel ranks after a row-parallel layer.
"""
import ctypes

import numpy as np

from . import _lib

CAAT_F32, CAAT_BF16 = 0, 1
CAAT_S_CONTIGUOUS, CAAT_S_RANDOM = 0, 1
CAAT_BWD_REDUCE_DOUT, CAAT_BWD_NO_REDUCE = 0, 1

__all__ = [
    "select_channels", "partial_channel_reduce", "rowpar_linear_fwd", "rowpar_linear_bwd",
    "rowpar_linear_bwd_workspace", "rowpar_linear_bwd_noalloc", "rowpar_linear_fwd_compact",
    "rowpar_linear_bwd_compact", "rowpar_linear_compact_workspace", "colpar_linear_fwd",
    "colpar_linear_bwd", "colpar_linear_bwd_workspace", "device_status", "last_kernel", "launch_count",
    "debug_set_wait", "CAAT_INJECT_NONE", "CAAT_INJECT_SKIP_LOADS", "pcr_pack", "pcr_unpack", "rank_fold",
    "CaatError", "CAAT_S_CONTIGUOUS", "CAAT_S_RANDOM", "CAAT_BWD_REDUCE_DOUT",
    "CAAT_BWD_NO_REDUCE",
]


class CaatError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.load().caat_status_string(status).decode()
        super().__init__("%s: %s" % (where, msg))


def _check(st: int, where: str):
    if st != 0:
        raise CaatError(st, where)


_TORCH = None


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return CAAT_F32
    if t.dtype == torch.bfloat16:
        return CAAT_BF16
    raise TypeError("caat: dtype must be float32 or bfloat16, got %s" % t.dtype)


def _stream_ptr(stream, like=None):
    """The CUDA stream handle: `stream`, else torch's current stream on the device
    of tensor `like` (read straight from torch's stream registry when it offers
    that, which is several times cheaper than building a Stream object)."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None and like is not None:
        return ctypes.c_void_p(raw(like.get_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _same_layout(ts, first, name):
    """Row stride shared by the 2-D tensors `ts` (all shaped, typed and strided like
    ts[0], which `_rowmajor` checks); raises otherwise."""
    ld = _rowmajor(ts[0], name)
    shp, st, dt = ts[0].shape, ts[0].stride(), ts[0].dtype
    for x in ts:
        if x.shape != shp or x.dtype != dt or not x.is_cuda:
            raise ValueError("caat: all %s tensors need one shape, dtype and device type" % name)
        if x.stride() != st and _rowmajor(x, name) != ld:
            raise ValueError("caat: all %s tensors need one row stride" % name)
    if first is not None and tuple(shp) != tuple(first):
        raise ValueError("caat: %s tensors must be %s" % (name, list(first)))
    return ld


def _rowmajor(t, name):
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("caat: %s must be 2-D with unit column stride" % name)
    if not t.is_cuda:
        raise ValueError("caat: %s must be a CUDA tensor" % name)
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _check_like(x, shape, dtype, name):
    """A tensor the library writes: it must have the shape and dtype the call
    implies, or the kernels would write past its end."""
    if tuple(x.shape) != tuple(shape) or x.dtype != dtype or not x.is_cuda:
        raise ValueError("caat: %s must be a CUDA tensor %s of dtype %s" % (name, list(shape), dtype))


def _workspace(workspace):
    """(pointer, bytes) of a caller's workspace tensor (contiguous, on the GPU)."""
    if workspace is None:
        return None, 0
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("caat: workspace must be a contiguous CUDA tensor")
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def _sel_ptr(sel):
    """S as a device index tensor, or an int n for the contiguous S = {0, ..., n-1}
    (passed to the library as a null pointer), or None for the empty set."""
    if sel is None:
        return None, 0
    if isinstance(sel, (int, np.integer)):
        if sel < 0:
            raise ValueError("caat: contiguous S size must be >= 0")
        return None, int(sel)
    if not sel.is_cuda or sel.dtype != _torch().int32 or sel.dim() != 1 or not sel.is_contiguous():
        raise ValueError("caat: sel must be a contiguous 1-D int32 CUDA tensor")
    return ctypes.c_void_p(sel.data_ptr() if sel.numel() else 0), sel.numel()


# --------------------------------------------------------------- channels

def select_channels(h: int, p: float, layout: int = CAAT_S_CONTIGUOUS, seed: int = 0) -> np.ndarray:
    """Sorted int32 indices of S, |S| = floor(p*h + 1/2) (host call)."""
    idx = np.zeros(max(int(h), 1), dtype=np.int32)
    n = ctypes.c_int64(0)
    st = _lib.load().caat_select_channels(int(h), float(p), int(layout),
                                           ctypes.c_uint64(int(seed) & (2**64 - 1)),
                                           idx.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n))
    _check(st, "caat_select_channels")
    return idx[: n.value].copy()


# ------------------------------------------------- partial channel-reduce

def partial_channel_reduce(ins, sel, outs=None, stream=None):
    """PCR over the t tensors ``ins`` (each [N, h], same shape/stride/dtype).

    Returns ``outs`` (allocated when None).  ``outs is ins`` (the same tensors)
    runs in place.
    """
    torch = _torch()
    t = len(ins)
    if t == 0:
        raise ValueError("caat: need at least one input")
    N, h = ins[0].shape
    ld_in = _same_layout(ins, None, "ins")
    if outs is None:
        outs = [torch.empty_like(x) for x in ins]
    if len(outs) != t:
        raise ValueError("caat: need as many outputs as inputs")
    ld_out = _same_layout(outs, (N, h), "outs")
    if outs[0].dtype != ins[0].dtype:
        raise ValueError("caat: outputs need the inputs' dtype")
    sp, ns = _sel_ptr(sel)
    st = _lib.load().caat_partial_channel_reduce(
        t, N, h, _dtype_code(ins[0]), _lib.ptr_array([x.data_ptr() for x in ins]), ld_in,
        _lib.ptr_array([y.data_ptr() for y in outs]), ld_out, sp, ns, _stream_ptr(stream, ins[0]))
    _check(st, "caat_partial_channel_reduce")
    return outs


# ---------------------------------------------------- row-parallel layer

def _weight_strides(W, K, h):
    if W.dim() != 2 or tuple(W.shape) != (K, h) or not W.is_cuda:
        raise ValueError("caat: W must be a CUDA tensor of logical shape [K, h] = [%d, %d]" % (K, h))
    return W.stride(0), W.stride(1)


def rowpar_linear_fwd(X, W, t: int, sel, outs=None, stream=None):
    """Row-parallel linear layer + PCR.  X [N, K]; W logical [K, h] (any strides,
    e.g. ``linear.weight.t()``).  Returns t tensors [N, h]."""
    torch = _torch()
    N, K = X.shape
    h = W.shape[1]
    ldx = _rowmajor(X, "X")
    w_rs, w_cs = _weight_strides(W, K, h)
    if W.dtype != X.dtype:
        raise TypeError("caat: X and W must share a dtype")
    if outs is None:
        outs = [torch.empty((N, h), dtype=X.dtype, device=X.device) for _ in range(t)]
    if len(outs) != t:
        raise ValueError("caat: need t output tensors")
    ldy = _same_layout(outs, (N, h), "outs")
    if outs[0].dtype != X.dtype:
        raise TypeError("caat: outputs must have X's dtype")
    sp, ns = _sel_ptr(sel)
    st = _lib.load().caat_rowpar_linear_fwd(
        int(t), N, K, h, _dtype_code(X), ctypes.c_void_p(X.data_ptr()), ldx,
        ctypes.c_void_p(W.data_ptr()), w_rs, w_cs,
        _lib.ptr_array([y.data_ptr() for y in outs]), ldy, sp, ns, _stream_ptr(stream, X))
    _check(st, "caat_rowpar_linear_fwd")
    return outs


def rowpar_linear_bwd_workspace(t: int, N: int, K: int, h: int, dtype_code: int, mode: int) -> int:
    return int(_lib.load().caat_rowpar_linear_bwd_workspace(int(t), int(N), int(K), int(h),
                                                            int(dtype_code), int(mode)))


def rowpar_linear_bwd(X, W, dOut, t: int, sel, mode: int = CAAT_BWD_REDUCE_DOUT,
                      dX=None, dW=None, workspace=None, stream=None):
    """Gradients of ``rowpar_linear_fwd``.  dOut: t tensors [N, h].
    Returns (dX [N, K], dW logical [K, h] with W's strides when allocated here)."""
    torch = _torch()
    N, K = X.shape
    h = W.shape[1]
    ldx = _rowmajor(X, "X")
    w_rs, w_cs = _weight_strides(W, K, h)
    if len(dOut) != t:
        raise ValueError("caat: need t upstream gradients")
    ldd = _same_layout(dOut, (N, h), "dOut")
    if dOut[0].dtype != X.dtype:
        raise TypeError("caat: dOut must have X's dtype")
    if W.dtype != X.dtype:
        raise TypeError("caat: X and W must share a dtype")
    if dX is None:
        dX = torch.empty((N, K), dtype=X.dtype, device=X.device)
    _check_like(dX, (N, K), X.dtype, "dX")
    lddx = _rowmajor(dX, "dX")
    if dW is None:
        if w_rs == 1:    # same layout as an nn.Linear weight: [h, K] storage
            dW = torch.empty((h, K), dtype=X.dtype, device=X.device).t()
        else:
            dW = torch.empty((K, h), dtype=X.dtype, device=X.device)
    _check_like(dW, (K, h), X.dtype, "dW")
    dw_rs, dw_cs = _weight_strides(dW, K, h)
    dt = _dtype_code(X)
    need = rowpar_linear_bwd_workspace(t, N, K, h, dt, mode)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    wp, wb = _workspace(workspace)
    sp, ns = _sel_ptr(sel)
    st = _lib.load().caat_rowpar_linear_bwd(
        int(t), N, K, h, dt, ctypes.c_void_p(X.data_ptr()), ldx,
        ctypes.c_void_p(W.data_ptr()), w_rs, w_cs,
        _lib.ptr_array([g.data_ptr() for g in dOut]), ldd,
        ctypes.c_void_p(dX.data_ptr()), lddx, ctypes.c_void_p(dW.data_ptr()), dw_rs, dw_cs,
        sp, ns, int(mode), wp, wb, _stream_ptr(stream, X))
    _check(st, "caat_rowpar_linear_bwd")
    return dX, dW


# ------------------------------------------------- compact outputs

def rowpar_linear_compact_workspace(t: int, N: int, K: int, h: int, dtype_code: int, index_list: bool,
                                    backward: bool) -> int:
    return int(_lib.load().caat_rowpar_linear_compact_workspace(int(t), int(N), int(K), int(h), int(dtype_code),
                                                                1 if index_list else 0, 1 if backward else 0))


def _compact_sel(sel, h):
    """(pointer, n_sel, whether it is an index list with 0 < |S| < h)."""
    sp, ns = _sel_ptr(sel)
    return sp, ns, (not isinstance(sel, (int, np.integer)) and sel is not None and 0 < ns < h)


def rowpar_linear_fwd_compact(X, W, t: int, sel, YS=None, YN=None, workspace=None, stream=None):
    """The fused layer with the outputs in compact form: YS [N, |S|] holds the
    channels of S once (the same on every rank), YN[r] [N, h - |S|] rank r's other
    channels, each in ascending channel order.  sel: an int n (S = the first n
    channels) or a device int32 index tensor; an index list needs a workspace (W
    in the S-first order), allocated here when None.  Returns (YS, YN)."""
    torch = _torch()
    N, K = X.shape
    h = W.shape[1]
    ldx = _rowmajor(X, "X")
    w_rs, w_cs = _weight_strides(W, K, h)
    if W.dtype != X.dtype:
        raise TypeError("caat: X and W must share a dtype")
    sp, n_sel, idx = _compact_sel(sel, h)
    if not 0 <= n_sel <= h:
        raise ValueError("caat: |S| must lie in [0, h]")
    if YS is None:
        YS = torch.empty((N, n_sel), dtype=X.dtype, device=X.device)
    if YN is None:
        YN = [torch.empty((N, h - n_sel), dtype=X.dtype, device=X.device) for _ in range(t)]
    if len(YN) != t:
        raise ValueError("caat: need t tensors YN")
    _check_like(YS, (N, n_sel), X.dtype, "YS")
    ldys = _rowmajor(YS, "YS") if YS.numel() else n_sel
    ldyn = _same_layout(YN, (N, h - n_sel), "YN") if h > n_sel and N > 0 else h - n_sel
    dt = _dtype_code(X)
    if workspace is None and idx:
        workspace = torch.empty(rowpar_linear_compact_workspace(t, N, K, h, dt, True, False),
                                dtype=torch.uint8, device=X.device)
    wp, wb = _workspace(workspace)
    st = _lib.load().caat_rowpar_linear_fwd_compact(
        int(t), N, K, h, dt, ctypes.c_void_p(X.data_ptr()), ldx,
        ctypes.c_void_p(W.data_ptr()), w_rs, w_cs,
        ctypes.c_void_p(YS.data_ptr()), ldys, _lib.ptr_array([y.data_ptr() for y in YN]), ldyn,
        sp, n_sel, wp, wb, _stream_ptr(stream, X))
    _check(st, "caat_rowpar_linear_fwd_compact")
    return YS, YN


def rowpar_linear_bwd_compact(X, W, dYS, dYN, t: int, sel=None, dX=None, dW=None, workspace=None, stream=None):
    """Gradients of ``rowpar_linear_fwd_compact``: dYS [N, |S|] (the gradient at YS,
    already summed over the ranks), dYN t tensors [N, h - |S|].  sel: as for the
    forward (None: the first dYS.shape[1] channels).  Returns (dX [N, K], dW
    logical [K, h] in the nn.Linear layout when allocated here).  workspace:
    allocated here when None (W in the S-first order for an index list, and the
    fp32 dW accumulator)."""
    torch = _torch()
    N, K = X.shape
    h = W.shape[1]
    if sel is None:
        sel = int(dYS.shape[1])
    sp, n_sel, idx = _compact_sel(sel, h)
    ldx = _rowmajor(X, "X")
    w_rs, w_cs = _weight_strides(W, K, h)
    if W.dtype != X.dtype or dYS.dtype != X.dtype:
        raise TypeError("caat: X, W and the gradients must share a dtype")
    if len(dYN) != t:
        raise ValueError("caat: need t tensors dYN")
    _check_like(dYS, (N, n_sel), X.dtype, "dYS")
    lddys = _rowmajor(dYS, "dYS") if dYS.numel() else n_sel
    lddyn = _same_layout(dYN, (N, h - n_sel), "dYN") if h > n_sel and N > 0 else h - n_sel
    if dX is None:
        dX = torch.empty((N, K), dtype=X.dtype, device=X.device)
    _check_like(dX, (N, K), X.dtype, "dX")
    lddx = _rowmajor(dX, "dX")
    if dW is None:
        dW = torch.empty((h, K), dtype=X.dtype, device=X.device).t()
    _check_like(dW, (K, h), X.dtype, "dW")
    dw_rs, dw_cs = _weight_strides(dW, K, h)
    dt = _dtype_code(X)
    if workspace is None:
        need = rowpar_linear_compact_workspace(t, N, K, h, dt, idx, True)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    wp, wb = _workspace(workspace)
    st = _lib.load().caat_rowpar_linear_bwd_compact(
        int(t), N, K, h, dt, ctypes.c_void_p(X.data_ptr()), ldx,
        ctypes.c_void_p(W.data_ptr()), w_rs, w_cs,
        ctypes.c_void_p(dYS.data_ptr()), lddys, _lib.ptr_array([g.data_ptr() for g in dYN]), lddyn,
        ctypes.c_void_p(dX.data_ptr()), lddx, ctypes.c_void_p(dW.data_ptr()), dw_rs, dw_cs,
        sp, n_sel, wp, wb, _stream_ptr(stream, X))
    _check(st, "caat_rowpar_linear_bwd_compact")
    return dX, dW


# ------------------------------------------------- column-parallel layer

def _rank_inputs(A, t: int, h: int, name: str):
    """t rank tensors [N, h] (a list, or a [t, N, h] tensor) sharing a row stride."""
    if not isinstance(A, (list, tuple)):
        if A.dim() != 3:
            raise ValueError("caat: %s must be t tensors [N, h] or one [t, N, h] tensor" % name)
        A = list(A.unbind(0))
    if len(A) != t:
        raise ValueError("caat: need t tensors in %s" % name)
    N = A[0].shape[0]
    ld = _same_layout(A, (N, h), name)
    return A, N, ld


def _w1_strides(W1, h, K, name="W1"):
    if W1.dim() != 2 or tuple(W1.shape) != (h, K) or not W1.is_cuda:
        raise ValueError("caat: %s must be a CUDA tensor of shape [h, K] = [%d, %d]" % (name, h, K))
    return W1.stride(0), W1.stride(1)


def colpar_linear_fwd(A, W1, t: int, Z=None, stream=None):
    """Column-parallel layer: A = the t ranks' inputs [N, h] (list or [t, N, h]
    tensor), W1 [h, K] (K-contiguous takes the tensor cores).  Returns Z [N, K]
    with column block r = A_r W1[:, block r]."""
    torch = _torch()
    h, K = W1.shape
    A, N, lda = _rank_inputs(A, t, h, "A")
    if W1.dtype != A[0].dtype:
        raise TypeError("caat: A and W1 must share a dtype")
    w1_rs, w1_cs = _w1_strides(W1, h, K)
    if Z is None:
        Z = torch.empty((N, K), dtype=W1.dtype, device=W1.device)
    if tuple(Z.shape) != (N, K) or Z.dtype != W1.dtype:
        raise ValueError("caat: Z must be [N, K] of W1's dtype")
    st = _lib.load().caat_colpar_linear_fwd(
        int(t), N, h, K, _dtype_code(W1), _lib.ptr_array([a.data_ptr() for a in A]), lda,
        ctypes.c_void_p(W1.data_ptr()), w1_rs, w1_cs, ctypes.c_void_p(Z.data_ptr()),
        _rowmajor(Z, "Z"), _stream_ptr(stream, W1))
    _check(st, "caat_colpar_linear_fwd")
    return Z


def colpar_linear_bwd_workspace(t: int, N: int, h: int, K: int, dtype_code: int) -> int:
    return int(_lib.load().caat_colpar_linear_bwd_workspace(int(t), int(N), int(h), int(K),
                                                            int(dtype_code)))


def colpar_linear_bwd(A, W1, dZ, t: int, sel, dA=None, dW1=None, workspace=None, stream=None):
    """Gradients of ``colpar_linear_fwd`` with the partial reduce on the input
    gradient: dA_r = PCR_S(dZ_r W1_r^T), dW1[:, block r] = A_r^T dZ_r.
    Returns (dA, dW1): dA a [t, N, h] tensor (or the list passed in), dW1 [h, K]
    with W1's strides when allocated here."""
    torch = _torch()
    h, K = W1.shape
    A, N, lda = _rank_inputs(A, t, h, "A")
    w1_rs, w1_cs = _w1_strides(W1, h, K)
    if tuple(dZ.shape) != (N, K) or dZ.dtype != W1.dtype:
        raise ValueError("caat: dZ must be [N, K] of W1's dtype")
    ldz = _rowmajor(dZ, "dZ")
    ret_dA = dA
    if dA is None:
        ret_dA = torch.empty((t, N, h), dtype=W1.dtype, device=W1.device)
    dAs, _, ldda = _rank_inputs(ret_dA, t, h, "dA")
    _check_like(dAs[0], (N, h), W1.dtype, "dA")
    if dW1 is None:
        dW1 = torch.empty_strided((h, K), W1.stride(), dtype=W1.dtype, device=W1.device)
    _check_like(dW1, (h, K), W1.dtype, "dW1")
    dw1_rs, dw1_cs = _w1_strides(dW1, h, K, "dW1")
    dt = _dtype_code(W1)
    if workspace is None:
        need = colpar_linear_bwd_workspace(t, N, h, K, dt)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=W1.device)
    wp, wb = _workspace(workspace)
    sp, ns = _sel_ptr(sel)
    st = _lib.load().caat_colpar_linear_bwd(
        int(t), N, h, K, dt, _lib.ptr_array([a.data_ptr() for a in A]), lda,
        ctypes.c_void_p(W1.data_ptr()), w1_rs, w1_cs, ctypes.c_void_p(dZ.data_ptr()), ldz,
        _lib.ptr_array([g.data_ptr() for g in dAs]), ldda,
        ctypes.c_void_p(dW1.data_ptr()), dw1_rs, dw1_cs, sp, ns, wp, wb, _stream_ptr(stream, W1))
    _check(st, "caat_colpar_linear_bwd")
    return ret_dA, dW1


# ------------------------------------ partial reduce across processes (steps)

def pcr_pack(Y, sel, P, stream=None):
    """P[:, i] = Y[:, S_i]: the channels of S of Y [N, h] into P [N, |S|]."""
    N, h = Y.shape
    sp, ns = _sel_ptr(sel)
    _check_like(P, (N, ns), Y.dtype, "P")
    st = _lib.load().caat_pcr_pack(N, h, _dtype_code(Y), ctypes.c_void_p(Y.data_ptr()), _rowmajor(Y, "Y"),
                                   sp, ns, ctypes.c_void_p(P.data_ptr()), _rowmajor(P, "P"),
                                   _stream_ptr(stream, Y))
    _check(st, "caat_pcr_pack")
    return P


def pcr_unpack(P, sel, Ys, stream=None):
    """Ys[k][:, S_i] = P[:, i] for every tensor of the list Ys (each [N, h])."""
    N, h = Ys[0].shape
    sp, ns = _sel_ptr(sel)
    _check_like(P, (N, ns), Ys[0].dtype, "P")
    ldy = _same_layout(Ys, (N, h), "Ys")
    st = _lib.load().caat_pcr_unpack(N, h, _dtype_code(P), ctypes.c_void_p(P.data_ptr()), _rowmajor(P, "P"),
                                     sp, ns, _lib.ptr_array([y.data_ptr() for y in Ys]), len(Ys), ldy,
                                     _stream_ptr(stream, P))
    _check(st, "caat_pcr_unpack")
    return Ys


def rank_fold(R, out, stream=None):
    """out = R[0] + R[1] + ... + R[t-1] (fp32 left fold in rank order, one rounding).
    R: contiguous [t, rows, cols]; out: [rows, cols]."""
    if R.dim() != 3 or not R.is_contiguous() or not R.is_cuda:
        raise ValueError("caat: R must be a contiguous CUDA tensor [t, rows, cols]")
    t, rows, cols = R.shape
    _check_like(out, (rows, cols), R.dtype, "out")
    st = _lib.load().caat_rank_fold(int(t), rows, cols, _dtype_code(R), ctypes.c_void_p(R.data_ptr()), cols,
                                    rows * cols, ctypes.c_void_p(out.data_ptr()), _rowmajor(out, "out"),
                                    _stream_ptr(stream, R))
    _check(st, "caat_rank_fold")
    return out


# ------------------------------------------------------------ diagnostics

def device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device-side error word."""
    return int(_lib.load().caat_get_device_status(_stream_ptr(stream)))


def last_kernel() -> str:
    return _lib.load().caat_last_kernel().decode()


def launch_count() -> int:
    return int(_lib.load().caat_launch_count())


CAAT_INJECT_NONE, CAAT_INJECT_SKIP_LOADS = 0, 1


def debug_set_wait(limit_ns: int = 0, inject: int = CAAT_INJECT_NONE) -> None:
    """Test hook of the failure path: the wait limit of the forward tile kernel's
    mbarrier waits (0 = the default 2 s) and an injected failure
    (CAAT_INJECT_SKIP_LOADS: its producer issues no load, so a wait runs out)."""
    _check(_lib.load().caat_debug_set_wait(int(limit_ns), int(inject)), "caat_debug_set_wait")


# ------------------------------------------- backward without a workspace

def rowpar_linear_bwd_noalloc(X, W, dOut, t: int, sel, mode: int = CAAT_BWD_REDUCE_DOUT,
                              dX=None, dW=None, stream=None):
    """``rowpar_linear_bwd`` for callers that cannot allocate device memory: the
    library's fixed 16 MiB scratch array replaces the workspace (the outputs dX
    and dW must then be passed in; nothing is allocated here).  Calls that overlap
    on the GPU race on that one array."""
    f = _lib.load().caat_rowpar_linear_bwd_noalloc
    if dX is None or dW is None:
        raise ValueError("caat: rowpar_linear_bwd_noalloc needs dX and dW passed in")
    N, K = X.shape
    h = W.shape[1]
    w_rs, w_cs = _weight_strides(W, K, h)
    if W.dtype != X.dtype:
        raise TypeError("caat: X and W must share a dtype")
    if len(dOut) != t:
        raise ValueError("caat: need t upstream gradients")
    ldd = _same_layout(dOut, (N, h), "dOut")
    if dOut[0].dtype != X.dtype:
        raise TypeError("caat: dOut must have X's dtype")
    _check_like(dX, (N, K), X.dtype, "dX")
    _check_like(dW, (K, h), X.dtype, "dW")
    dw_rs, dw_cs = _weight_strides(dW, K, h)
    sp, ns = _sel_ptr(sel)
    st = f(int(t), N, K, h, _dtype_code(X), ctypes.c_void_p(X.data_ptr()), _rowmajor(X, "X"),
           ctypes.c_void_p(W.data_ptr()), w_rs, w_cs,
           _lib.ptr_array([g.data_ptr() for g in dOut]), ldd,
           ctypes.c_void_p(dX.data_ptr()), _rowmajor(dX, "dX"),
           ctypes.c_void_p(dW.data_ptr()), dw_rs, dw_cs, sp, ns, int(mode), _stream_ptr(stream))
    _check(st, "caat_rowpar_linear_bwd_noalloc")
    return dX, dW
