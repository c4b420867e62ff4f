"""Planted mistakes: each test builds a copy of the CPU oracle with one plausible
slip and checks that the pins of tests/test_oracle.py would catch it.  This shows
the pins are tight (a pin that a wrong oracle also passes pins nothing).

Mutants are compiled from the oracle's C source with a textual edit on the CPU;
nothing here touches the GPU or the product library."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

from oracle import build as obuild

SRC = open(obuild.SRC).read()


def _mutant(old, new):
    assert SRC.count(old) >= 1, old
    src = SRC.replace(old, new, 1)
    d = tempfile.mkdtemp(prefix="caat_mutant_")
    c = os.path.join(d, "m.c")
    so = os.path.join(d, "m.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True)
    L = ctypes.CDLL(so)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    L.orc_rowpar_fwd.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, I64, P, P]
    L.orc_rowpar_bwd.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, P, I64, ctypes.c_int, P, P]
    L.orc_select_channels.argtypes = [I64, ctypes.c_double, ctypes.c_int, ctypes.c_uint64, P, P]
    L.orc_pcr_f32.argtypes = [ctypes.c_int, I64, I64, P, P, I64, P]
    L.orc_pcr_f32.restype = I64
    return L


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fwd(L, X, W, t, S):
    N, K = X.shape
    h = W.shape[1]
    out = np.empty((t, N, h))
    macs = np.zeros(1, dtype=np.int64)
    S = np.ascontiguousarray(S, dtype=np.int32)
    L.orc_rowpar_fwd(t, N, K, h, _p(X), _p(W), _p(S), S.size, _p(out), _p(macs))
    return out


def _bwd(L, X, W, G, t, S, mode):
    N, K = X.shape
    h = W.shape[1]
    dX = np.empty((N, K))
    dW = np.empty((K, h))
    S = np.ascontiguousarray(S, dtype=np.int32)
    L.orc_rowpar_bwd(t, N, K, h, _p(X), _p(W), _p(G), _p(S), S.size, mode, _p(dX), _p(dW))
    return dX, dW


def _case(seed=0, t=3, N=4, K=9, h=7):
    r = np.random.default_rng(seed)
    return (np.ascontiguousarray(r.standard_normal((N, K))), np.ascontiguousarray(r.standard_normal((K, h))),
            np.ascontiguousarray(r.standard_normal((t, N, h))), t)


def _fwd_pins_hold(L):
    """p = 1 and p = 0 pins of the forward (numpy matmul)."""
    X, W, _, t = _case()
    K = X.shape[1]
    kt = K // t
    full = _fwd(L, X, W, t, np.arange(W.shape[1]))
    ok1 = all(np.allclose(full[r], X @ W, rtol=1e-12, atol=1e-12) for r in range(t))
    ens = _fwd(L, X, W, t, [])
    ok0 = all(np.allclose(ens[r], X[:, r * kt:(r + 1) * kt] @ W[r * kt:(r + 1) * kt], rtol=1e-12, atol=1e-12)
              for r in range(t))
    return ok1 and ok0


def _bwd_pins_hold(L):
    """Finite differences of sum_r <G_r, Out_r> (reduce-dOut mode) at a mixed S."""
    X, W, G, t = _case(1)
    S = np.array([0, 2, 5], dtype=np.int32)
    dX, dW = _bwd(L, X, W, G, t, S, 0)
    eps = 1e-3

    def loss(Xv, Wv):
        return float(np.sum(_fwd(L, Xv, Wv, t, S) * G))

    for idx in [(0, 0), (1, 4), (3, 8)]:
        Xp = X.copy(); Xp[idx] += eps
        Xm = X.copy(); Xm[idx] -= eps
        if abs((loss(Xp, W) - loss(Xm, W)) / (2 * eps) - dX[idx]) > 1e-7:
            return False
    for idx in [(0, 0), (4, 2), (8, 6)]:
        Wp = W.copy(); Wp[idx] += eps
        Wm = W.copy(); Wm[idx] -= eps
        if abs((loss(X, Wp) - loss(X, Wm)) / (2 * eps) - dW[idx]) > 1e-7:
            return False
    return True


def test_unmutated_oracle_passes_the_same_checks():
    L = _mutant("int orc_rowpar_fwd(", "int orc_rowpar_fwd(")   # identity edit
    assert _fwd_pins_hold(L)
    assert _bwd_pins_hold(L)


@pytest.mark.parametrize("old,new", [
    # shard offset off by one k
    ("for (int64_t k = (int64_t)r * kt; k < (int64_t)(r + 1) * kt; ++k)\n                    acc += X[n * K + k] * W[k * h + c];",
     "for (int64_t k = (int64_t)r * kt + 1; k < (int64_t)(r + 1) * kt; ++k)\n                    acc += X[n * K + k] * W[k * h + c];"),
    # W indexed transposed
    ("acc += X[n * K + k] * W[k * h + c];", "acc += X[n * K + k] * W[c * K + k];"),
    # the reduce drops the last rank
    ("for (int q = 1; q < t; ++q) acc = acc + Y[((int64_t)q * N + n) * h + c];\n                for (int r = 0; r < t; ++r) Out[((int64_t)r * N + n) * h + c] = acc;\n                reduced += 1;\n            } else {\n                for (int r = 0; r < t; ++r)\n                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];\n            }\n        }\n    }\n    free(inS);\n    return reduced;\n}\n\n/* ------------------------------------------------ row-parallel",
     "for (int q = 1; q < t - 1; ++q) acc = acc + Y[((int64_t)q * N + n) * h + c];\n                for (int r = 0; r < t; ++r) Out[((int64_t)r * N + n) * h + c] = acc;\n                reduced += 1;\n            } else {\n                for (int r = 0; r < t; ++r)\n                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];\n            }\n        }\n    }\n    free(inS);\n    return reduced;\n}\n\n/* ------------------------------------------------ row-parallel"),
    # non-S channels scaled by t
    ("                for (int r = 0; r < t; ++r)\n                    Out[((int64_t)r * N + n) * h + c] = Y[((int64_t)r * N + n) * h + c];\n            }\n        }\n    }\n    free(inS);\n    return reduced;\n}\n\n/* ------------------------------------------------ row-parallel",
     "                for (int r = 0; r < t; ++r)\n                    Out[((int64_t)r * N + n) * h + c] = t * Y[((int64_t)r * N + n) * h + c];\n            }\n        }\n    }\n    free(inS);\n    return reduced;\n}\n\n/* ------------------------------------------------ row-parallel"),
])
def test_forward_mutants_are_caught(old, new):
    assert not _fwd_pins_hold(_mutant(old, new))


@pytest.mark.parametrize("old,new", [
    # backward forgets the reduce (uses G as is in the reduce mode)
    ("    if (mode == 0)\n        orc_pcr_f64(t, N, h, G, sel, n_sel, dY);",
     "    if (mode == 7)\n        orc_pcr_f64(t, N, h, G, sel, n_sel, dY);"),
    # dW from the wrong rank's gradient
    ("acc += X[n * K + k] * dY[((int64_t)r * N + n) * h + c];",
     "acc += X[n * K + k] * dY[((int64_t)((r + 1) % t) * N + n) * h + c];"),
    # dX with W transposed
    ("for (int64_t c = 0; c < h; ++c) acc += g[c] * W[k * h + c];",
     "for (int64_t c = 0; c < h; ++c) acc += g[c] * W[(c % K) * h + (k % h)];"),
])
def test_backward_mutants_are_caught(old, new):
    assert not _bwd_pins_hold(_mutant(old, new))


def test_biased_shuffle_mutant_is_caught():
    # j = next mod h instead of mod (i + 1): the uniformity pin must fail
    L = _mutant("uint64_t j = sm64_next(&st) % (uint64_t)(i + 1);", "uint64_t j = sm64_next(&st) % (uint64_t)h;")
    counts = {}
    n = 6000
    idx = np.zeros(3, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int64)
    for seed in range(n):
        L.orc_select_channels(3, 1 / 3, 1, seed, _p(idx), _p(cnt))
        a = int(idx[0])
        L.orc_select_channels(3, 2 / 3, 1, seed, _p(idx), _p(cnt))
        b = sorted(set(idx[:2].tolist()) - {a})[0]
        counts[(a, b)] = counts.get((a, b), 0) + 1
    exp = n / 6
    chi2 = sum((c - exp) ** 2 / exp for c in counts.values()) + exp * (6 - len(counts))
    assert chi2 >= 20.5


# ------------------------------------------------ column-parallel backward

def _colpar_bwd_from(L):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    L.orc_colpar_bwd.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, P, I64, P, P]

    def bwd(A, W1, dZ, t, S):
        A = np.ascontiguousarray(A, dtype=np.float64)
        W1 = np.ascontiguousarray(W1, dtype=np.float64)
        dZ = np.ascontiguousarray(dZ, dtype=np.float64)
        _, N, h = A.shape
        K = W1.shape[1]
        S = np.ascontiguousarray(S, dtype=np.int32)
        dA = np.empty((t, N, h))
        dW1 = np.empty((h, K))
        L.orc_colpar_bwd(t, N, h, K, _p(A), _p(W1), _p(dZ), _p(S), S.size, _p(dA), _p(dW1))
        return dA, dW1
    return bwd


def _colpar_pins_hold(L):
    from tests.test_oracle_colpar import colpar_logical_fd_errors
    bwd = _colpar_bwd_from(L)
    return all(colpar_logical_fd_errors(bwd, t, N, h, K, p, seed) <= 1e-8
               for (t, N, h, K, p, seed) in [(3, 2, 5, 6, 0.4, 5), (2, 2, 4, 4, 1.0, 6)])


def test_unmutated_colpar_passes_the_same_checks():
    assert _colpar_pins_hold(_mutant("int orc_colpar_bwd(", "int orc_colpar_bwd("))


@pytest.mark.parametrize("old,new", [
    # the input gradient is not reduced at all
    ("orc_pcr_f64(t, N, h, P, sel, n_sel, dA);",
     "memcpy(dA, P, sizeof(double) * (size_t)((int64_t)t * N * h));"),
    # every rank's input gradient taken over all of K (a full reduce for every channel)
    ("for (int64_t k = (int64_t)r * kt; k < (int64_t)(r + 1) * kt; ++k)\n                    acc += dZ[n * K + k] * W1[c * K + k];",
     "for (int64_t k = 0; k < K; ++k)\n                    acc += dZ[n * K + k] * W1[c * K + k];"),
    # dW1 from the wrong rank's input
    ("acc += A[((int64_t)r * N + n) * h + c] * dZ[n * K + k];",
     "acc += A[((int64_t)((r + 1) % t) * N + n) * h + c] * dZ[n * K + k];"),
])
def test_colpar_mutants_are_caught(old, new):
    assert not _colpar_pins_hold(_mutant(old, new))
