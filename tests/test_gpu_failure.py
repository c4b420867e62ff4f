"""Device-side failure detection of the forward tile kernel, exercised without a
GPU fault: a test hook makes the kernel's TMA producer issue no load, so the MMA
issuer's wait for its first operands can never complete.  With a 1 ms wait limit
that wait gives up, the kernel records CAAT_ERR_TIMEOUT and exits (no copy and
no MMA is in flight: none was issued), and caat_get_device_status reports it.
The same context then runs the normal path again and matches the oracle."""
import numpy as np
import pytest

import caat_inputs as ci
from oracle import oracle as orc
from tests.gpu_helpers import TOL, dev, host_values, rel_fro, sel_dev, to_f64, torch

pytestmark = pytest.mark.gpu

CAAT_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def caat():
    import partial_activation_sync_gb300 as m
    return m


# one CTA per tile (k_t = 64), and a CTA pair (k_t = 512, two row blocks)
@pytest.mark.parametrize("cluster,kt", [("1", 64), ("2", 512)])
def test_forward_wait_timeout_reported_then_context_usable(caat, cluster, kt, monkeypatch):
    T = torch()
    monkeypatch.setenv("CAAT_FWD_CLUSTER", cluster)
    monkeypatch.setenv("CAAT_FWD_SKINNY", "0")      # the tile kernel (the few-token one takes N <= 256)
    t, N, h = 2, 256, 256
    X = ci.normal(1901, (N, kt * t))
    Wl = ci.normal(1902, (kt * t, h), std=0.02)
    S = caat.select_channels(h, 0.5, caat.CAAT_S_RANDOM, 19)
    Xd = dev(X, "bf16")
    Wd = dev(np.ascontiguousarray(Wl.T), "bf16").t()
    sel = sel_dev(S)
    assert caat.device_status() == 0
    caat.debug_set_wait(1_000_000, caat.CAAT_INJECT_SKIP_LOADS)
    try:
        caat.rowpar_linear_fwd(Xd, Wd, t, sel)
        kernel = caat.last_kernel()
        status = caat.device_status()
    finally:
        caat.debug_set_wait(0, caat.CAAT_INJECT_NONE)
    assert kernel == "rowpar_fwd_tc"
    assert status == CAAT_ERR_TIMEOUT
    assert caat.device_status() == 0          # reading the status cleared it
    # the context is still usable: the same call now runs to completion
    outs = caat.rowpar_linear_fwd(Xd, Wd, t, sel)
    T.cuda.synchronize()
    assert caat.device_status() == 0
    want, _ = orc.rowpar_fwd(host_values(X, "bf16"), host_values(Wl, "bf16"), t, S)
    for r in range(t):
        assert rel_fro(to_f64(outs[r]), want[r]) <= TOL["bf16"]
