"""NumPy front end of the CPU oracle for CAAT-Net's partial channel-reduce.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may call this module; the product library never does.  It shares no
code with the CUDA path.  The arithmetic lives in ``caat_oracle.c`` (naive loops,
double accumulation); this file only marshals NumPy arrays through ctypes.

Every function follows "Tensor-Parallelism with Partially Synchronized
Activations" (NeurIPS 2025), Introduction, the paragraph that defines the partial
channel-reduce (a subset S of hidden channels is summed over the t tensor-parallel
ranks, the rest stay rank-local; S empty = ensemble, S full = vanilla all-reduce;
forward and backward must agree).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_get_threads.restype = ctypes.c_int
        L.orc_splitmix64.argtypes = [ctypes.c_uint64, _i64, _p]
        L.orc_select_channels.argtypes = [_i64, ctypes.c_double, ctypes.c_int,
                                          ctypes.c_uint64, _p, _p]
        L.orc_select_channels.restype = ctypes.c_int
        L.orc_f32_to_bf16.argtypes = [_i64, _p, _p]
        for name in ("orc_pcr_f32", "orc_pcr_bf16", "orc_pcr_f64"):
            f = getattr(L, name)
            f.argtypes = [ctypes.c_int, _i64, _i64, _p, _p, _i64, _p]
            f.restype = _i64
        L.orc_rowpar_fwd.argtypes = [ctypes.c_int, _i64, _i64, _i64, _p, _p, _p,
                                     _i64, _p, _p]
        L.orc_rowpar_fwd.restype = ctypes.c_int
        L.orc_rowpar_bwd.argtypes = [ctypes.c_int, _i64, _i64, _i64, _p, _p, _p,
                                     _p, _i64, ctypes.c_int, _p, _p]
        L.orc_rowpar_bwd.restype = ctypes.c_int
        L.orc_colpar_fwd.argtypes = [ctypes.c_int, _i64, _i64, _i64, _p, _p, _p]
        L.orc_colpar_fwd.restype = ctypes.c_int
        L.orc_colpar_bwd.argtypes = [ctypes.c_int, _i64, _i64, _i64, _p, _p, _p, _p, _i64,
                                     _p, _p]
        L.orc_colpar_bwd.restype = ctypes.c_int
        _LIB = L
    return _LIB


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ------------------------------------------------------------------ helpers

def splitmix64(seed: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.uint64)
    lib().orc_splitmix64(ctypes.c_uint64(seed & (2**64 - 1)), n, _ptr(out))
    return out


def f32_to_bf16(a) -> np.ndarray:
    """Round float32 to bf16 words (nearest, ties to even) -- the oracle's own rounding."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16(a.size, _ptr(a), _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Widen bf16 words exactly (a bf16 value is the top half of an fp32 word)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------ channel selection

def select_channels(h: int, p: float, layout: int = 0, seed: int = 0) -> np.ndarray:
    """Sorted int32 indices of S: |S| = floor(p*h + 1/2); layout 0 = first |S|
    channels, layout 1 = first |S| of a splitmix64-driven Fisher-Yates shuffle."""
    idx = np.zeros(max(h, 1), dtype=np.int32)
    n = np.zeros(1, dtype=np.int64)
    rc = lib().orc_select_channels(h, float(p), int(layout),
                                   ctypes.c_uint64(seed & (2**64 - 1)), _ptr(idx), _ptr(n))
    if rc != 0:
        raise ValueError("orc_select_channels: invalid argument")
    return idx[: int(n[0])].copy()


# --------------------------------------------------- partial channel-reduce

def _sel(sel):
    return np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1))


def pcr_f32(Y, sel):
    """Y float32 [t, N, h] -> (Out float32 [t, N, h], reduced element count)."""
    Y = np.ascontiguousarray(Y, dtype=np.float32)
    t, N, h = Y.shape
    s = _sel(sel)
    out = np.empty_like(Y)
    red = lib().orc_pcr_f32(t, N, h, _ptr(Y), _ptr(s), s.size, _ptr(out))
    return out, int(red)


def pcr_bf16(Y, sel):
    """Y bf16 words uint16 [t, N, h] -> (Out uint16 [t, N, h], reduced count)."""
    Y = np.ascontiguousarray(Y, dtype=np.uint16)
    t, N, h = Y.shape
    s = _sel(sel)
    out = np.empty_like(Y)
    red = lib().orc_pcr_bf16(t, N, h, _ptr(Y), _ptr(s), s.size, _ptr(out))
    return out, int(red)


def pcr_f64(Y, sel):
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    t, N, h = Y.shape
    s = _sel(sel)
    out = np.empty_like(Y)
    red = lib().orc_pcr_f64(t, N, h, _ptr(Y), _ptr(s), s.size, _ptr(out))
    return out, int(red)


# ------------------------------------------------- row-parallel linear layer

def rowpar_fwd(X, W, t: int, sel):
    """X [N, K], W [K, h] (float64, logical layout) -> (Out [t, N, h] f64, MACs)."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    N, K = X.shape
    K2, h = W.shape
    assert K == K2
    s = _sel(sel)
    out = np.empty((t, N, h), dtype=np.float64)
    macs = np.zeros(1, dtype=np.int64)
    rc = lib().orc_rowpar_fwd(t, N, K, h, _ptr(X), _ptr(W), _ptr(s), s.size,
                              _ptr(out), _ptr(macs))
    if rc != 0:
        raise ValueError("orc_rowpar_fwd: invalid argument")
    return out, int(macs[0])


REDUCE_DOUT = 0
NO_REDUCE = 1


def rowpar_bwd(X, W, G, t: int, sel, mode: int = REDUCE_DOUT):
    """X [N, K], W [K, h], G [t, N, h] (float64) -> (dX [N, K], dW [K, h])."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    G = np.ascontiguousarray(G, dtype=np.float64)
    N, K = X.shape
    _, h = W.shape
    assert G.shape == (t, N, h)
    s = _sel(sel)
    dX = np.empty((N, K), dtype=np.float64)
    dW = np.empty((K, h), dtype=np.float64)
    rc = lib().orc_rowpar_bwd(t, N, K, h, _ptr(X), _ptr(W), _ptr(G), _ptr(s),
                              s.size, int(mode), _ptr(dX), _ptr(dW))
    if rc != 0:
        raise ValueError("orc_rowpar_bwd: invalid argument")
    return dX, dW


# ---------------------------------------------- column-parallel linear layer

def colpar_fwd(A, W1, t: int):
    """A [t, N, h] (rank r's own input), W1 [h, K] (float64) -> Z [N, K], column
    block r = A_r W1[:, block r]."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    W1 = np.ascontiguousarray(W1, dtype=np.float64)
    t2, N, h = A.shape
    h2, K = W1.shape
    assert t2 == t and h2 == h
    Z = np.empty((N, K), dtype=np.float64)
    if lib().orc_colpar_fwd(t, N, h, K, _ptr(A), _ptr(W1), _ptr(Z)) != 0:
        raise ValueError("orc_colpar_fwd: invalid argument")
    return Z


def colpar_bwd(A, W1, dZ, t: int, sel):
    """A [t, N, h], W1 [h, K], dZ [N, K] (float64) -> (dA [t, N, h], dW1 [h, K]);
    dA = PCR over S of the ranks' dZ_r W1_r^T."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    W1 = np.ascontiguousarray(W1, dtype=np.float64)
    dZ = np.ascontiguousarray(dZ, dtype=np.float64)
    _, N, h = A.shape
    K = W1.shape[1]
    assert dZ.shape == (N, K)
    s = _sel(sel)
    dA = np.empty((t, N, h), dtype=np.float64)
    dW1 = np.empty((h, K), dtype=np.float64)
    if lib().orc_colpar_bwd(t, N, h, K, _ptr(A), _ptr(W1), _ptr(dZ), _ptr(s), s.size,
                            _ptr(dA), _ptr(dW1)) != 0:
        raise ValueError("orc_colpar_bwd: invalid argument")
    return dA, dW1
