"""The autograd front ends with their options combined: leading dimensions,
masks, num_label_tokens, the saved-lse / no-lse / one-pass CE backward and the
recomputing / eager FLCE, against the fp64 oracle (bars of the other parity
tests: loss 1e-3 relative, gradients 2e-2 max relative and 5e-3 normwise)."""
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lh():
    import lm_head_linear_fwd_gb300 as m
    return m


def _grad_ok(got, want):
    assert oracle.max_rel_err(got.float().cpu(), want) <= 2e-2
    assert oracle.normwise_err(got.float().cpu(), want) <= 5e-3


@pytest.mark.parametrize("mode", ["saved", "no_lse", "eager", "eager_inplace"])
@pytest.mark.parametrize("reduction,nlt", [("mean", None), ("sum", 700)])
def test_ce_logits_options(lh, mode, reduction, nlt):
    B, T, V = 3, 41, 5003
    p = wl.random_ce(B * T, V, torch.bfloat16, seed=101, ignore_frac=0.05)
    mask = (torch.arange(B * T) % 7 != 3).to(torch.int64)
    labels = torch.where(mask == 0, torch.full_like(p.labels, -100), p.labels)
    want_loss = oracle.ce_forward(p.logits, labels, -100, reduction, nlt)["loss"]
    want = oracle.ce_backward(p.logits, labels, -100, reduction, nlt, grad_loss=0.25)
    x = p.logits.cuda().reshape(B, T, V).contiguous().requires_grad_(True)
    kw = dict(reduction=reduction, num_label_tokens=nlt, mask=mask.cuda().reshape(B, T))
    if mode == "no_lse":
        kw["save_lse"] = False
    if mode.startswith("eager"):
        kw["eager"] = True
        kw["inplace_grad"] = mode == "eager_inplace"
    loss = lh.ce_logits(x, p.labels.cuda().reshape(B, T), **kw)
    (0.25 * loss).backward()
    torch.cuda.synchronize()
    assert abs(loss.item() - want_loss) <= 1e-3 * abs(want_loss)
    assert x.grad.shape == (B, T, V)
    _grad_ok(x.grad.reshape(B * T, V), want)


@pytest.mark.parametrize("eager", [False, True])
def test_flce_options(lh, eager):
    B, T, D, V = 2, 150, 128, 3001
    p = wl.random_flce(B * T, D, V, torch.bfloat16, bias=True, seed=102, w_std=0.05)
    mask = (torch.arange(B * T) % 5 != 0).to(torch.int64)
    labels = torch.where(mask == 0, torch.full_like(p.labels, -100), p.labels)
    ref = oracle.flce_forward(p.H, p.W, p.bias, labels, -100, "mean")
    gr = oracle.flce_backward(p.H, p.W, p.bias, labels, -100, "mean", grad_loss=2.0)
    H = p.H.cuda().reshape(B, T, D).requires_grad_(True)
    W = p.W.cuda().requires_grad_(True)
    b = p.bias.cuda().requires_grad_(True)
    loss = lh.flce(H, W, p.labels.cuda().reshape(B, T), b, reduction="mean",
                   mask=mask.cuda().reshape(B, T), eager=eager, chunk=128)
    (2.0 * loss).backward()
    torch.cuda.synchronize()
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    assert H.grad.shape == (B, T, D)
    _grad_ok(H.grad.reshape(B * T, D), gr["grad_H"])
    _grad_ok(W.grad, gr["grad_W"])
    _grad_ok(b.grad, gr["grad_b"])
