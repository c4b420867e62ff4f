"""GPU parity of the column-parallel layer (forward; backward with the partial
reduce on the input gradient) against the CPU oracle (double accumulation).

Tolerances are relative Frobenius errors, max over Z, the t rank input gradients
and dW1: 1e-5 for fp32 (FFMA) and 1e-2 for bf16 inputs with fp32 accumulation.
The S channels of the input gradient must be bit-identical across ranks."""
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


def _w1(W32, dtype, layout):
    """Device W1 [h, K]: 'rm' = stored row-major (K contiguous, the tensor-core
    layout), 'cm' = stored [K, h] and passed transposed."""
    if layout == "rm":
        return dev(W32, dtype)
    return dev(np.ascontiguousarray(W32.T), dtype).t()


def _inputs(t, N, h, K, seed):
    A = ci.normal(1200 + seed, (t, N, h))
    W1 = ci.normal(2200 + seed, (h, K), std=0.02)
    dZ = ci.normal(3200 + seed, (N, K))
    return A, W1, dZ


def _run(caat, t, N, h, K, p, layout_S, dtype, wl="rm", seed=0):
    A, W1, dZ = _inputs(t, N, h, K, seed)
    S = caat.select_channels(h, p, layout_S, 4200 + seed)
    Ad = dev(A, dtype)
    W1d = _w1(W1, dtype, wl)
    Z = caat.colpar_linear_fwd(Ad, W1d, t)
    fwd_kernel = caat.last_kernel()
    dA, dW1 = caat.colpar_linear_bwd(Ad, W1d, dev(dZ, dtype), t, sel_dev(S))
    bwd_kernel = caat.last_kernel()
    torch().cuda.synchronize()
    assert caat.device_status() == 0
    hA, hW, hZ = host_values(A, dtype), host_values(W1, dtype), host_values(dZ, dtype)
    wZ = orc.colpar_fwd(hA, hW, t)
    wA, wW = orc.colpar_bwd(hA, hW, hZ, t, S)
    got = (to_f64(Z), np.stack([to_f64(dA[r]) for r in range(t)]), to_f64(dW1))
    # S as an index list: the S channels of dA may fold the ranks' rounded
    # partials dZ_r W1_r^T (the tile kernel); their magnitudes bound that rounding
    spread = None
    if 0 < S.size < h and t > 1:
        parts, _ = orc.colpar_bwd(hA, hW, hZ, t, np.zeros(0, np.int32))
        spread = np.zeros(wA.shape[1:])
        spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    return got, (wZ, wA, wW, spread), S, (fwd_kernel, bwd_kernel)


def _check(got, want, S, t, dtype):
    gZ, gA, gW = got
    wZ, wA, wW, spread = want
    check(gZ, wZ, dtype)
    for r in range(t):
        check(gA[r], wA[r], dtype, what=r, spread=spread)
    check(gW, wW, dtype)
    for r in range(1, t):
        assert np.array_equal(gA[r][:, S], gA[0][:, S])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("t,N,h,kt", [(1, 5, 24, 8), (2, 7, 40, 4), (3, 129, 200, 96), (8, 33, 72, 16)])
@pytest.mark.parametrize("wl", ["rm", "cm"])
def test_colpar_small_shapes(caat, dtype, t, N, h, kt, wl):
    for p in (0.0, 0.5, 1.0):
        for layout in (0, 1):
            got, want, S, _ = _run(caat, t, N, h, kt * t, p, layout, dtype, wl, seed=t + N)
            _check(got, want, S, t, dtype)


@pytest.mark.parametrize("t,N,h,K", [(8, 256, 768, 2304), (8, 300, 768, 3072), (3, 200, 520, 408),
                                     (4, 130, 256, 256),
                                     (4, 384, 520, 1024)])   # k_t = 256: the GEMMs on CTA pairs
@pytest.mark.parametrize("p,layout", [(0.5, 0), (0.5, 1), (0.0, 0), (1.0, 0)])
def test_colpar_tensor_core_shapes(caat, t, N, h, K, p, layout):
    got, want, S, kernels = _run(caat, t, N, h, K, p, layout, "bf16", "rm", seed=N)
    _check(got, want, S, t, "bf16")
    # the tensor-core kernels ran (no fallback to the CUDA-core GEMMs)
    assert kernels[0] == "rowpar_bwd_dx_tc"
    assert kernels[1] in ("rowpar_fwd_tc", "rowpar_fwd_skinny_tc")


def test_colpar_contiguous_set_by_size(caat):
    # S passed as a size (null index list) against the index list of the same S:
    # dW1 and the channels of dA outside S are computed alike (the same bits); the
    # S channels of dA are summed in fp32 over all of K (size) or folded from the
    # ranks' rounded partials (index list), and both match the oracle
    t, N, h, K = 8, 256, 768, 3072
    A, W1, dZ = _inputs(t, N, h, K, 9)
    Ad, W1d, dZd = dev(A, "bf16"), dev(W1, "bf16"), dev(dZ, "bf16")
    dA1, dW1a = caat.colpar_linear_bwd(Ad, W1d, dZd, t, 384)
    dA2, dW1b = caat.colpar_linear_bwd(Ad, W1d, dZd, t, sel_dev(np.arange(384)))
    torch().cuda.synchronize()
    assert bool((dW1a == dW1b).all())
    assert bool((dA1[:, :, 384:] == dA2[:, :, 384:]).all())
    hA, hW, hZ = host_values(A, "bf16"), host_values(W1, "bf16"), host_values(dZ, "bf16")
    S = np.arange(384, dtype=np.int32)
    wA, _ = orc.colpar_bwd(hA, hW, hZ, t, S)
    parts, _ = orc.colpar_bwd(hA, hW, hZ, t, np.zeros(0, np.int32))
    spread = np.zeros((N, h))
    spread[:, S] = np.abs(parts).sum(axis=0)[:, S]
    for r in range(t):
        check(to_f64(dA1[r]), wA[r], "bf16")
        check(to_f64(dA2[r]), wA[r], "bf16", spread=spread)


def test_colpar_empty_sizes(caat):
    T = torch()
    t, h, K = 2, 8, 4
    A = T.zeros((t, 0, h), device="cuda")
    W1 = T.ones((h, K), device="cuda")
    Z = caat.colpar_linear_fwd(A, W1, t)
    dA, dW1 = caat.colpar_linear_bwd(A, W1, T.zeros((0, K), device="cuda"), t, 4)
    T.cuda.synchronize()
    assert Z.shape == (0, K) and dA.shape == (t, 0, h)
    assert bool((dW1 == 0).all())       # empty sum over tokens


def test_colpar_full_size_sampled(caat):
    # The 130M MLP up-projection at full size (N = 8 x 1024 tokens, h = 768,
    # FFN 3072, t = 8, p = 0.5) in the launch configuration the benchmark times;
    # the oracle checks sampled token rows of Z and dA (rows are independent) and
    # sampled columns of dW1 in every block (columns are independent).
    t, N, h, K = 8, 8192, 768, 3072
    A, W1, dZ = _inputs(t, N, h, K, 17)
    Ad, W1d, dZd = dev(A, "bf16"), dev(W1, "bf16"), dev(dZ, "bf16")
    Z = caat.colpar_linear_fwd(Ad, W1d, t)
    dA, dW1 = caat.colpar_linear_bwd(Ad, W1d, dZd, t, 384)
    torch().cuda.synchronize()
    assert caat.device_status() == 0
    hA, hW, hZ = host_values(A, "bf16"), host_values(W1, "bf16"), host_values(dZ, "bf16")
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(N, 48, replace=False))
    S = np.arange(384)
    wZ = orc.colpar_fwd(hA[:, rows], hW, t)
    wA, _ = orc.colpar_bwd(hA[:, rows], hW, hZ[rows], t, S)
    gZ = to_f64(Z)[rows]
    check(gZ, wZ, "bf16")
    gA = to_f64(dA)[:, rows]
    for r in range(t):
        check(gA[r], wA[r], "bf16")
    kt = K // t
    cols = np.concatenate([r * kt + np.sort(rng.choice(kt, 4, replace=False)) for r in range(t)])
    _, wW = orc.colpar_bwd(hA, hW[:, cols], hZ[:, cols], t, S)
    check(to_f64(dW1)[:, cols], wW, "bf16")
