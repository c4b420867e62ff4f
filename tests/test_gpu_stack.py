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


def _run(model, tokens):
    """Loss (float) and gradients (float64, CPU) of one forward + backward."""
    T = torch()
    import partial_activation_sync_gb300 as caat
    model.zero_grad(set_to_none=True)
    loss = model(tokens)
    loss.backward()
    T.cuda.synchronize()
    assert caat.device_status() == 0
    return float(loss.detach()), {n: p.grad.double().cpu().numpy() for n, p in model.named_parameters()}


@pytest.mark.parametrize("layout", ["contiguous", "random"])
@pytest.mark.parametrize("placement", ["reduce_dout", "column"])
def test_stack_loss_and_gradients_match_reference(placement, layout):
    """S contiguous (the layers get its size) or a seeded random subset (the
    layers get an index list); the reference takes the same S."""
    T = torch()
    from oracle import stack as ost
    from partial_activation_sync_gb300.caatnet import CAATNet
    T.manual_seed(1234)
    t, heads, layers, seq, batch, vocab = 8, 16, 2, 64, 2, 1024
    model = CAATNet(vocab=vocab, h=768, heads=heads, layers=layers, ffn=3072, t=t, p=0.5, seq=seq,
                    placement=placement, layout=layout, seed=31)
    model = model.cuda().to(T.bfloat16)
    assert (model.sel_idx is None) == (layout == "contiguous")
    tokens = T.from_numpy(np.random.default_rng(7).integers(0, vocab, (batch, seq))).cuda()
    got_L, got_g = _run(model, tokens)
    params = {n: p.detach().double().cpu() for n, p in model.named_parameters()}
    s = model.n_sel if layout == "contiguous" else model.S
    L, grads = ost.loss_and_grads(params, tokens.cpu(), t, heads, layers, s, placement)
    assert abs(got_L - L) <= 1e-3 * abs(L), (got_L, L)
    for name in got_g:
        assert rel_fro(got_g[name], grads[name].numpy()) <= 2e-2, name


@pytest.mark.parametrize("placement", ["reduce_dout", "column"])
def test_relabelled_model_matches_random_set(placement):
    """relabel_channels: the model with a random S and its relabelled copy (S the
    first |S| channels, passed by size) give the same loss, and the same gradients
    once renamed, within the bounds above (the two run different kernels, so they
    round differently)."""
    T = torch()
    from partial_activation_sync_gb300.caatnet import CAATNet, relabel_channels
    T.manual_seed(77)
    t, heads, layers, seq, batch, vocab = 8, 16, 2, 64, 2, 1024
    model = CAATNet(vocab=vocab, h=768, heads=heads, layers=layers, ffn=3072, t=t, p=0.5, seq=seq,
                    placement=placement, layout="random", seed=5).cuda().to(T.bfloat16)
    relab, perm = relabel_channels(model)
    assert relab.sel_idx is None and relab.n_sel == model.n_sel
    assert np.array_equal(np.sort(perm[:model.n_sel]), model.S)
    tokens = T.from_numpy(np.random.default_rng(8).integers(0, vocab, (batch, seq))).cuda()
    L_r, g_r = _run(model, tokens)
    L_c, g_c = _run(relab, tokens)
    assert abs(L_r - L_c) <= 1e-3 * abs(L_r), (L_r, L_c)
    for name, g in g_r.items():
        if name == "emb":
            g = g[:, perm]
        else:
            g = g[perm]          # gains, biases and the four weights: rows
        assert rel_fro(g_c[name], g) <= 2e-2, name


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
