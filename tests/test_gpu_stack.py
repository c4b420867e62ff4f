"""The CAAT-Net block stack on the GPU (row-parallel layers in this library's
kernels, the rest PyTorch) against the float64 CPU reference of the stack.

Both placements of the backward reduce are checked, each against the reference's
matching placement.  Reduced stack: 2 layers, sequence 64, batch 2, vocabulary
1024, with the 130M model's width (h = 768, 16 heads, FFN 3072), t = 8, p = 0.5.
Tolerances are relative. The parameters and every activation are bf16, so each op
rounds to 2^-9 relative; through two blocks, forward and backward, the measured
relative Frobenius error of the parameter gradients is at most 0.0078 (about four
bf16 roundings' worth; both placements, seeds 1234 and 99) and that of the loss
4.2e-5.  The bounds are 2e-2 on gradients (2.5 times the largest seen, about ten
roundings) and 1e-3 on the loss."""
import numpy as np
import pytest

from tests.gpu_helpers import rel_fro, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tensor_cores_only(monkeypatch):
    """Every layer of the stack takes a tensor-core kernel: no CUDA-core opt-in."""
    monkeypatch.delenv("CAAT_ALLOW_FALLBACK", raising=False)


@pytest.mark.parametrize("placement", ["reduce_dout", "column"])
def test_stack_loss_and_gradients_match_reference(placement):
    T = torch()
    from oracle import stack as ost
    from partial_activation_sync_gb300.caatnet import CAATNet
    import partial_activation_sync_gb300 as caat
    T.manual_seed(1234)
    t, heads, layers, seq, batch, vocab = 8, 16, 2, 64, 2, 1024
    model = CAATNet(vocab=vocab, h=768, heads=heads, layers=layers, ffn=3072, t=t, p=0.5, seq=seq,
                    placement=placement)
    model = model.cuda().to(T.bfloat16)
    tokens = T.from_numpy(np.random.default_rng(7).integers(0, vocab, (batch, seq))).cuda()
    loss = model(tokens)
    loss.backward()
    T.cuda.synchronize()
    assert caat.device_status() == 0
    params = {n: p.detach().double().cpu() for n, p in model.named_parameters()}
    L, grads = ost.loss_and_grads(params, tokens.cpu(), t, heads, layers, model.n_sel, placement)
    assert abs(float(loss.detach()) - L) <= 1e-3 * abs(L), (float(loss.detach()), L)
    for name, p in model.named_parameters():
        g = p.grad.double().cpu().numpy()
        assert rel_fro(g, grads[name].numpy()) <= 2e-2, name


@pytest.mark.parametrize("placement", ["reduce_dout", "column"])
def test_stack_training_step_runs(placement):
    T = torch()
    from partial_activation_sync_gb300.caatnet import CAATNet, train_step
    T.manual_seed(5)
    model = CAATNet(vocab=512, h=768, heads=16, layers=1, ffn=3072, t=8, p=0.5, seq=128,
                    placement=placement).cuda().to(T.bfloat16)
    opt = T.optim.AdamW(model.parameters(), lr=1e-3)
    tokens = T.randint(0, 512, (2, 128), device="cuda")
    l0 = float(train_step(model, opt, tokens))
    for _ in range(5):
        l1 = float(train_step(model, opt, tokens))
    assert np.isfinite(l0) and np.isfinite(l1) and l1 < l0   # overfits one batch
