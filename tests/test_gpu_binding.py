"""The Python binding refuses output tensors whose shape or dtype differs from
what the call writes (the kernels would otherwise write past their end), before
it calls the library."""
import pytest

from tests.gpu_helpers import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


def test_rowpar_backward_output_checks(caat):
    T = torch()
    t, N, K, h = 2, 16, 128, 64
    X = T.zeros((N, K), dtype=T.float32, device="cuda")
    W = T.zeros((K, h), dtype=T.float32, device="cuda")
    G = [T.zeros((N, h), dtype=T.float32, device="cuda") for _ in range(t)]
    n0 = caat.launch_count()
    with pytest.raises(ValueError, match="dX"):        # bf16 dX for an fp32 layer
        caat.rowpar_linear_bwd(X, W, G, t, 8, dX=T.zeros((N, K), dtype=T.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="dX"):        # too few columns
        caat.rowpar_linear_bwd(X, W, G, t, 8, dX=T.zeros((N, K // 2), dtype=T.float32, device="cuda"))
    with pytest.raises(ValueError, match="dW"):
        caat.rowpar_linear_bwd(X, W, G, t, 8, dW=T.zeros((K, h), dtype=T.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="workspace"):
        caat.rowpar_linear_bwd(X, W, G, t, 8, workspace=T.zeros((64, 64), dtype=T.uint8, device="cuda").t())
    with pytest.raises(TypeError):
        caat.rowpar_linear_bwd(X, W.to(T.bfloat16), G, t, 8)
    dX = T.zeros((N, K), dtype=T.float32, device="cuda")
    dW = T.zeros((K, h), dtype=T.float32, device="cuda")
    with pytest.raises(ValueError):                     # one gradient short
        caat.rowpar_linear_bwd_noalloc(X, W, G[:1], t, 8, dX=dX, dW=dW)
    with pytest.raises(ValueError, match="dW"):
        caat.rowpar_linear_bwd_noalloc(X, W, G, t, 8, dX=dX, dW=dW[:, : h // 2])
    assert caat.launch_count() == n0
    # the same call with fitting outputs runs
    caat.rowpar_linear_bwd(X, W, G, t, 8, dX=dX, dW=dW)
    T.cuda.synchronize()
    assert caat.device_status() == 0


def test_colpar_backward_output_checks(caat):
    T = torch()
    t, N, h, K = 2, 16, 64, 128
    A = T.zeros((t, N, h), dtype=T.bfloat16, device="cuda")
    W1 = T.zeros((h, K), dtype=T.bfloat16, device="cuda")
    dZ = T.zeros((N, K), dtype=T.bfloat16, device="cuda")
    n0 = caat.launch_count()
    with pytest.raises(ValueError, match="dA"):
        caat.colpar_linear_bwd(A, W1, dZ, t, 8, dA=T.zeros((t, N, h), dtype=T.float32, device="cuda"))
    with pytest.raises(ValueError, match="dW1"):
        caat.colpar_linear_bwd(A, W1, dZ, t, 8, dW1=T.zeros((h, K), dtype=T.float32, device="cuda"))
    assert caat.launch_count() == n0
