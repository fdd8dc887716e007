"""Edge cases of both paths against the oracle: degenerate sizes, K/V/N tails
that are not multiples of any tile, logits far outside exp's range, labels at
the last column, ignore_index inside the vocabulary.  Tolerances as in
tests/test_gpu_flce.py and tests/test_gpu_ce_logits.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lh():
    import lm_head_linear_fwd_gb300 as m
    return m


def _grad_ok(got, want, name, mr_tol=2e-2, nw_tol=5e-3):
    mr = oracle.max_rel_err(got.float().cpu(), want)
    nw = oracle.normwise_err(got.float().cpu(), want)
    assert mr <= mr_tol and nw <= nw_tol, (name, mr, nw)


def _flce_all(lh, H, W, b, y, reduction="sum", nlt=None, chunk=None, ignore_index=-100):
    out = lh.flce_fwd(H.cuda(), W.cuda(), y.cuda(), None if b is None else b.cuda(), ignore_index,
                      reduction, nlt)
    bw = lh.flce_bwd(H.cuda(), W.cuda(), y.cuda(), out.lse, out.n_valid,
                     torch.ones(1, device="cuda"), None if b is None else b.cuda(), ignore_index,
                     reduction, nlt, chunk)
    fo, fb = lh.flce_fwd_bwd(H.cuda(), W.cuda(), y.cuda(), None if b is None else b.cuda(),
                             ignore_index, reduction, nlt, chunk)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    lh.check_status(fo.status)
    return out, bw, fo, fb


def _compare(H, W, b, y, res, reduction="sum", nlt=None, ignore_index=-100):
    out, bw, fo, fb = res
    ref = oracle.flce_forward(H, W, b, y, ignore_index, reduction, nlt)
    gr = oracle.flce_backward(H, W, b, y, ignore_index, reduction, nlt)
    for o in (out, fo):
        assert int(o.n_valid.item()) == ref["n_valid"]
        assert abs(o.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"]) + 1e-6
    for g in (bw, fb):
        _grad_ok(g.grad_H, gr["grad_H"], "grad_H")
        _grad_ok(g.grad_W, gr["grad_W"], "grad_W")
        if b is not None:
            _grad_ok(g.grad_bias, gr["grad_b"], "grad_b")


@pytest.mark.parametrize("N,D,V", [(1, 64, 1000), (5, 8, 7), (300, 72, 250), (130, 200, 257),
                                   (257, 136, 513)])
def test_flce_odd_sizes(lh, N, D, V):
    p = wl.random_flce(N, D, V, torch.bfloat16, bias=True, seed=N * 31 + D, ignore_frac=0.1,
                       w_std=0.1)
    if N > 3:
        p.labels[0] = V - 1
    res = _flce_all(lh, p.H, p.W, p.bias, p.labels)
    _compare(p.H, p.W, p.bias, p.labels, res)


def test_flce_single_class(lh):
    """V = 1: every valid row has loss 0 and zero gradients."""
    p = wl.random_flce(64, 32, 1, torch.bfloat16, seed=5, ignore_frac=0.2)
    p.labels[p.labels != -100] = 0
    out, bw, fo, fb = _flce_all(lh, p.H, p.W, None, p.labels, "mean")
    for o in (out, fo):
        assert abs(o.loss.item()) <= 1e-6
    for g in (bw, fb):
        assert float(g.grad_H.float().abs().max()) <= 1e-6
        assert float(g.grad_W.abs().max()) <= 1e-6


def test_flce_huge_logits(lh):
    """Logits of magnitude ~100 (exp would overflow fp32 without the max shift)."""
    p = wl.random_flce(200, 64, 3000, torch.bfloat16, seed=9, w_std=1.5)
    res = _flce_all(lh, p.H, p.W, None, p.labels)
    assert float(p.H.float().abs().max() * p.W.float().abs().max()) > 10
    out = res[0]
    assert math.isfinite(out.loss.item())
    _compare(p.H, p.W, None, p.labels, res)


def test_flce_ignore_index_inside_vocab(lh):
    p = wl.random_flce(256, 64, 1000, torch.bfloat16, seed=11, ignore_frac=0.0)
    p.labels[::5] = 17
    res = _flce_all(lh, p.H, p.W, None, p.labels, "mean", ignore_index=17)
    _compare(p.H, p.W, None, p.labels, res, "mean", ignore_index=17)


def test_ce_extreme_logits(lh):
    """+-3e4 logits and -inf entries: lse stays finite and exact to tolerance."""
    V = 777
    x = torch.randn(16, V) * 5
    x[0, 3] = 30000.0
    x[1, :] = -30000.0
    x[1, 9] = -29990.0
    x[2, 100:200] = float("-inf")
    logits = x.to(torch.bfloat16)
    y = torch.tensor([3, 9, 5] + [1] * 13)
    out = lh.ce_logits_fwd(logits.cuda(), y.cuda(), want_rows=True)
    grad = lh.ce_logits_bwd(logits.cuda(), y.cuda(), out.lse, out.n_valid,
                            torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    ref = oracle.ce_forward(logits, y)
    lse = out.lse.cpu().double().numpy()
    assert np.all(np.abs(lse - ref["lse"]) <= 5e-5 * (1 + np.abs(ref["lse"])))
    dz = oracle.ce_backward(logits, y)
    _grad_ok(grad, dz, "dlogits")
    assert torch.all(grad[2, 100:200] == 0)


def test_ce_single_column(lh):
    logits = torch.randn(40, 1).to(torch.bfloat16)
    y = torch.zeros(40, dtype=torch.int64)
    y[::4] = -100
    out = lh.ce_logits_fwd(logits.cuda(), y.cuda(), -100, "mean")
    grad = lh.ce_logits_bwd(logits.cuda(), y.cuda(), out.lse, out.n_valid,
                            torch.ones(1, device="cuda"), -100, "mean")
    torch.cuda.synchronize()
    assert abs(out.loss.item()) <= 1e-6 and out.n_valid.item() == 30
    assert float(grad.float().abs().max()) <= 1e-6


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_flce_one_valid_row(lh, reduction):
    # every row ignored but one: the loss is that row's, every other row's
    # gradient is zero, and grad_W / grad_b come from that row alone
    p = wl.random_flce(300, 128, 2000, torch.bfloat16, bias=True, seed=61, ignore_frac=0.0)
    y = torch.full_like(p.labels, -100)
    y[137] = 1999  # in the last, partial vocabulary tile
    res = _flce_all(lh, p.H, p.W, p.bias, y, reduction)
    _compare(p.H, p.W, p.bias, y, res, reduction)
    out, bw, fo, fb = res
    assert int(out.n_valid.item()) == 1
    for g in (bw, fb):
        gh = g.grad_H.float().cpu()
        assert torch.count_nonzero(torch.cat([gh[:137], gh[138:]])) == 0


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_ce_one_valid_row(lh, reduction):
    p = wl.random_ce(200, 5000, torch.bfloat16, seed=62, ignore_frac=0.0)
    logits = p.logits.cuda()
    y = torch.full_like(p.labels, -100)
    y[3] = 4999
    out = lh.ce_logits_fwd(logits, y.cuda(), -100, reduction)
    g = torch.ones(1, device="cuda")
    for lse in (out.lse, None):
        grad = lh.ce_logits_bwd(logits, y.cuda(), lse, out.n_valid, g, -100, reduction)
        torch.cuda.synchronize()
        lh.check_status(out.status)
        ref = oracle.ce_forward(p.logits, y, -100, reduction)
        assert int(out.n_valid.item()) == 1
        assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
        _grad_ok(grad, oracle.ce_backward(p.logits, y, -100, reduction), "dlogits")
        gc = grad.float().cpu()
        assert torch.count_nonzero(torch.cat([gc[:3], gc[4:]])) == 0


def test_leading_dimensions_are_rows(lh):
    # logits [B, T, V] / H [B, T, D] with labels [B, T]: the same results as the
    # flattened call, and gradients in the input's shape
    c = wl.random_ce(2 * 48, 3000, torch.bfloat16, seed=71)
    x2 = c.logits.cuda().requires_grad_(True)
    l2 = lh.ce_logits(x2, c.labels.cuda(), reduction="mean")
    l2.backward()
    x3 = c.logits.cuda().reshape(2, 48, 3000).requires_grad_(True)
    l3 = lh.ce_logits(x3, c.labels.cuda().reshape(2, 48), reduction="mean")
    l3.backward()
    assert torch.equal(l2, l3) and x3.grad.shape == (2, 48, 3000)
    assert torch.equal(x3.grad.reshape(96, 3000), x2.grad)
    p = wl.random_flce(2 * 128, 128, 2000, torch.bfloat16, seed=72)
    H2 = p.H.cuda().requires_grad_(True)
    W2 = p.W.cuda().requires_grad_(True)
    lh.flce(H2, W2, p.labels.cuda(), reduction="sum").backward()
    H3 = p.H.cuda().reshape(2, 128, 128).requires_grad_(True)
    W3 = p.W.cuda().requires_grad_(True)
    lh.flce(H3, W3, p.labels.cuda().reshape(2, 128), reduction="sum").backward()
    assert H3.grad.shape == (2, 128, 128)
    assert torch.equal(H3.grad.reshape(256, 128), H2.grad) and torch.equal(W3.grad, W2.grad)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_flce_empty_batch(lh, dtype):
    # N = 0: loss 0, n_valid 0, no grad_H rows, grad_W and grad_bias zero
    # (grad_W left as it is when accumulating); every call path
    V, D = 1000, 128
    W = torch.randn(V, D, device="cuda").to(dtype)
    b = torch.randn(V, device="cuda").to(dtype)
    H = torch.empty(0, D, dtype=dtype, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    out = lh.flce_fwd(H, W, y, b, -100, "mean")
    gW = torch.full((V, D), float("nan"), device="cuda")
    gb = torch.full((V,), float("nan"), device="cuda")
    bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b, -100,
                     "mean", grad_W=gW, grad_bias=gb)
    acc = torch.ones(V, D, device="cuda")
    lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b, -100, "mean",
                want_grad_H=False, want_grad_bias=False, grad_W=acc, accumulate_grad_W=True)
    fo, fr = lh.flce_fwd_bwd(H, W, y, b, -100, "sum")
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert out.loss.item() == 0.0 and out.n_valid.item() == 0
    assert bw.grad_H.shape == (0, D)
    assert torch.count_nonzero(gW) == 0 and torch.count_nonzero(gb) == 0
    assert torch.all(acc == 1.0)
    assert fo.loss.item() == 0.0 and fo.n_valid.item() == 0
    assert torch.count_nonzero(fr.grad_W) == 0 and torch.count_nonzero(fr.grad_bias) == 0
    Hr = H.clone().requires_grad_(True)
    Wr = W.clone().requires_grad_(True)
    loss = lh.flce(Hr, Wr, y, reduction="sum")
    loss.backward()
    assert loss.item() == 0.0 and Hr.grad.shape == (0, D)
    assert torch.count_nonzero(Wr.grad) == 0
