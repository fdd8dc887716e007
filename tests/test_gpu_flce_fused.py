"""Fused forward + backward (flce_fwd_bwd, 6NDV) against the fp64 oracle and
against the recomputing path (flce_fwd + flce_bwd).

Same tolerances as tests/test_gpu_flce.py (tests/tolerances.py): loss 1e-3
relative, per-row lse 2e-5 (1 + |lse|) for bf16 (the tf32 cut added for fp32
inputs), n_valid exact, gradients 2e-2 max-relative / 5e-3 normwise.
The logits are kept between the two halves as bf16 offsets from each tile's
maximum, one more rounding than the recomputing path, still inside those bars.
"""
import numpy as np
import pytest
import torch

import oracle
import tolerances as tol
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lh():
    import lm_head_linear_fwd_gb300 as m
    return m


def _to(p):
    b = p.bias.cuda() if p.bias is not None else None
    return p.H.cuda(), p.W.cuda(), b, p.labels.cuda()


def _grad_ok(got, want, name):
    mr = oracle.max_rel_err(got.float().cpu(), want)
    nw = oracle.normwise_err(got.float().cpu(), want)
    assert mr <= 2e-2 and nw <= 5e-3, (name, mr, nw)


def _fused(lh, p, chunk=None, g=None, accumulate_init=None):
    H, W, b, y = _to(p)
    gw = accumulate_init.cuda().clone() if accumulate_init is not None else None
    gl = torch.tensor([g], device="cuda") if g is not None else None
    out, bw = lh.flce_fwd_bwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, chunk, gl,
                              want_rows=True, grad_W=gw,
                              accumulate_grad_W=accumulate_init is not None)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    return out, bw


def _check(p, out, bw, g=1.0, grad_W_init=None):
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens)
    assert int(out.n_valid.item()) == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"]) + 1e-6
    tol.check_flce_lse(out.lse, ref["lse"], p.H, p.W, p.bias)
    if out.loss_rows is not None:
        tol.check_flce_loss_rows(out.loss_rows, ref["loss_rows"], ref["lse"], p.H, p.W)
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens,
                              grad_loss=g, grad_W_init=grad_W_init)
    _grad_ok(bw.grad_H, gr["grad_H"], "grad_H")
    _grad_ok(bw.grad_W, gr["grad_W"], "grad_W")
    if p.bias is not None:
        _grad_ok(bw.grad_bias, gr["grad_b"], "grad_b")


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_fused_tiny_fp32(lh, reduction):
    p = wl.tiny_flce(reduction)
    out, bw = _fused(lh, p, g=1.5)
    _check(p, out, bw, g=1.5)


def test_fused_small_model(lh):
    p = wl.small_flce()
    out, bw = _fused(lh, p)
    _check(p, out, bw)


@pytest.mark.parametrize("N,D,V,chunk,bias,dtype", [
    (700, 256, 3001, 256, True, torch.bfloat16),
    (129, 64, 777, 128, False, torch.bfloat16),
    (300, 96, 1234, 128, True, torch.float32),
])
def test_fused_ragged_multi_chunk(lh, N, D, V, chunk, bias, dtype):
    p = wl.random_flce(N, D, V, dtype, bias=bias, seed=N + 7, reduction="mean")
    out, bw = _fused(lh, p, chunk=chunk, g=0.5)
    _check(p, out, bw, g=0.5)


def test_fused_accumulate_and_num_label_tokens(lh):
    p = wl.random_flce(256, 128, 1000, torch.bfloat16, seed=43, num_label_tokens=200)
    init = torch.randn(1000, 128) * 0.01
    out, bw = _fused(lh, p, accumulate_init=init)
    _check(p, out, bw, grad_W_init=init.double().numpy())


@pytest.mark.parametrize("reduction,nlt", [("mean", None), ("sum", 0)])
def test_fused_zero_guards(lh, reduction, nlt):
    p = wl.random_flce(150, 64, 500, torch.bfloat16, bias=True, seed=63, reduction=reduction,
                       num_label_tokens=nlt)
    if nlt is None:
        p.labels[:] = -100
    out, bw = _fused(lh, p)
    assert out.loss.item() == 0.0
    for t in (bw.grad_H, bw.grad_W, bw.grad_bias):
        assert torch.count_nonzero(t).item() == 0


def test_fused_autograd_eager(lh):
    p = wl.random_flce(300, 128, 2000, torch.bfloat16, bias=True, seed=83, reduction="mean")
    H, W, b, y = _to(p)
    for t in (H, W, b):
        t.requires_grad_(True)
    loss = lh.flce(H, W, y, b, reduction="mean", chunk=128, eager=True)
    (loss * 2.5).backward()
    torch.cuda.synchronize()
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, "mean", grad_loss=2.5)
    _grad_ok(H.grad, gr["grad_H"], "grad_H")
    _grad_ok(W.grad, gr["grad_W"], "grad_W")
    _grad_ok(b.grad, gr["grad_b"], "grad_b")


def test_fused_deterministic(lh):
    p = wl.random_flce(600, 256, 5000, torch.bfloat16, bias=True, seed=103)
    o1, b1 = _fused(lh, p, chunk=256)
    o2, b2 = _fused(lh, p, chunk=256)
    assert torch.equal(o1.loss, o2.loss) and torch.equal(o1.lse, o2.lse)
    for a, c in ((b1.grad_H, b2.grad_H), (b1.grad_W, b2.grad_W), (b1.grad_bias, b2.grad_bias)):
        assert torch.equal(a, c)


def test_fused_matches_recompute_path_at_full_size(lh):
    """Llama3-8B shape: the fused call against flce_fwd + flce_bwd (checked
    against the oracle elsewhere), and sampled rows against the oracle."""
    p = wl.llama3_8b_flce(device="cuda")
    H, W, y = p.H, p.W, p.labels
    out, bw = lh.flce_fwd_bwd(H, W, y, None, -100, p.reduction, p.num_label_tokens,
                              want_rows=True)
    ref_o = lh.flce_fwd(H, W, y, None, -100, p.reduction, p.num_label_tokens, want_rows=True)
    ref_b = lh.flce_bwd(H, W, y, ref_o.lse, ref_o.n_valid, torch.ones(1, device="cuda"), None,
                        -100, p.reduction, p.num_label_tokens)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert out.n_valid.item() == ref_o.n_valid.item()
    assert abs(out.loss.item() - ref_o.loss.item()) <= 1e-5 * abs(ref_o.loss.item())
    assert torch.allclose(out.lse, ref_o.lse, rtol=0, atol=1e-4)
    for a, c, n in ((bw.grad_H, ref_b.grad_H, "grad_H"), (bw.grad_W, ref_b.grad_W, "grad_W")):
        nw = oracle.normwise_err(a.float().cpu(), c.float().cpu().double().numpy())
        assert nw <= 5e-3, (n, nw)
    rows = np.sort(np.random.default_rng(3).choice(p.N, 16, replace=False))
    W64 = p.W.cpu().double().numpy()
    gr = oracle.flce_backward(p.H.cpu(), W64, None, p.labels.cpu(), -100, p.reduction,
                              p.num_label_tokens, rows=rows, want_grad_W=False,
                              n_valid_total=int(out.n_valid.item()))
    _grad_ok(bw.grad_H[torch.as_tensor(rows, device="cuda")], gr["grad_H"], "grad_H rows")
