"""Cross-entropy on given logits: CUDA path through the C ABI vs the fp64 oracle.

Tolerances (the loss and gradient bars of the hot-path specification, plus
what the arithmetic gives):
* loss: |gpu - ref| <= 1e-3 |ref| (fp32 per-row lse, fp64 reduction; the
  observed error is far smaller);
* per-row lse: |gpu - ref| <= 5e-5 (1 + |ref|): fp32 sums of up to 1.3e5
  terms, each from ex2.approx (relative error ~2^-22);
* n_valid and the gathered label logit: exact;
* dlogits (bf16 output): max relative <= 2e-2 and normwise <= 5e-3 (one bf16
  rounding, 2^-9 relative, per element).
"""
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


def _dev(p):
    return p.logits.cuda(), p.labels.cuda()


def _check_fwd(out, ref, rows=None):
    torch.cuda.synchronize()
    lse = out.lse.cpu().double().numpy()
    want = ref["lse"]
    if rows is not None:
        lse = lse[rows]
    assert np.all(np.abs(lse - want) <= 5e-5 * (1 + np.abs(want))), np.max(np.abs(lse - want))


def _check_grad(got, want):
    assert oracle.max_rel_err(got.float().cpu(), want) <= 2e-2
    assert oracle.normwise_err(got.float().cpu(), want) <= 5e-3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("reduction,nlt", [("sum", None), ("mean", None), ("sum", 1000)])
@pytest.mark.parametrize("N,V,ld", [(300, 1000, 1000), (77, 1003, 1011), (5, 32777, 32777),
                                    (130, 4099, 4099), (64, 50257, 50257), (9, 128255, 128255)])
def test_ce_parity(lh, dtype, reduction, nlt, N, V, ld):
    p = wl.random_ce(N, V, dtype, seed=N + V, reduction=reduction, num_label_tokens=nlt, ld=ld)
    logits, labels = _dev(p)
    out = lh.ce_logits_fwd(logits, labels, -100, reduction, nlt, want_rows=True,
                           want_label_logit=True)
    ref = oracle.ce_forward(p.logits, p.labels, -100, reduction, nlt)
    _check_fwd(out, ref)
    assert int(out.n_valid.item()) == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    zl = out.label_logit.cpu().double().numpy()
    valid = p.labels.numpy() != -100
    assert np.array_equal(zl[valid], ref["label_logit"][valid])  # exact widening
    assert np.all(np.isnan(zl[~valid]))
    g = torch.tensor([0.7], device="cuda")
    grad = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, g, -100, reduction, nlt)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, reduction, nlt, grad_loss=0.7))


def test_inplace_grad_aliases_logits(lh):
    p = wl.random_ce(64, 5000, torch.bfloat16, seed=3)
    base, labels = _dev(p)
    base = base.contiguous().requires_grad_(True)
    logits = base * 1.0  # a non-leaf, like the output of an lm_head
    seen = {}
    logits.register_hook(lambda g: seen.setdefault("g", g))
    loss = lh.ce_logits(logits, labels, inplace_grad=True)
    loss.backward()
    torch.cuda.synchronize()
    # the gradient handed to autograd is the logits storage itself
    assert seen["g"].data_ptr() == logits.data_ptr()
    _check_grad(seen["g"], oracle.ce_backward(p.logits, p.labels))
    assert torch.equal(logits.detach(), seen["g"])
    _check_grad(base.grad, oracle.ce_backward(p.logits, p.labels))


def test_default_does_not_mutate_logits(lh):
    p = wl.random_ce(32, 3000, torch.bfloat16, seed=4)
    logits = p.logits.cuda().contiguous().requires_grad_(True)
    before = logits.detach().clone()
    lh.ce_logits(logits, p.labels.cuda()).backward()
    torch.cuda.synchronize()
    assert torch.equal(logits.detach(), before)
    assert logits.grad.data_ptr() != logits.data_ptr()


def test_second_inplace_backward_raises(lh):
    p = wl.random_ce(8, 300, torch.bfloat16, seed=5)
    logits = p.logits.cuda().contiguous().requires_grad_(True)
    loss = lh.ce_logits(logits, p.labels.cuda(), inplace_grad=True)
    loss.backward(retain_graph=True)
    with pytest.raises(RuntimeError):
        loss.backward()


def test_double_backward_raises(lh):
    p = wl.random_ce(8, 300, torch.float32, seed=6)
    logits = p.logits.cuda().contiguous().requires_grad_(True)
    loss = lh.ce_logits(logits, p.labels.cuda())
    (g,) = torch.autograd.grad(loss, logits, create_graph=True)
    with pytest.raises(RuntimeError):
        g.sum().backward()


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_all_ignored(lh, reduction):
    logits = torch.randn(16, 500, device="cuda").bfloat16()
    labels = torch.full((16,), -100, dtype=torch.int64, device="cuda")
    out = lh.ce_logits_fwd(logits, labels, -100, reduction)
    grad = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, torch.ones(1, device="cuda"),
                            -100, reduction)
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and out.n_valid.item() == 0
    assert torch.count_nonzero(grad).item() == 0


def test_zero_num_label_tokens(lh):
    p = wl.random_ce(16, 700, torch.bfloat16, seed=8)
    logits, labels = _dev(p)
    out = lh.ce_logits_fwd(logits, labels, -100, "sum", 0)
    grad = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, torch.ones(1, device="cuda"),
                            -100, "sum", 0)
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and out.n_valid.item() == int((p.labels != -100).sum())
    assert torch.count_nonzero(grad).item() == 0


def test_bad_label_sets_status_and_row_is_ignored(lh):
    p = wl.random_ce(20, 600, torch.bfloat16, seed=9, ignore_frac=0.0)
    logits, labels = _dev(p)
    labels[3] = 600  # out of range
    labels[7] = -5
    out = lh.ce_logits_fwd(logits, labels, -100, "mean")
    grad = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, torch.ones(1, device="cuda"),
                            -100, "mean")
    torch.cuda.synchronize()
    assert int(out.status.item()) == -5
    with pytest.raises(lh.FlceError):
        lh.check_status(out.status)
    ref_labels = p.labels.clone()
    ref_labels[3] = -100
    ref_labels[7] = -100
    ref = oracle.ce_forward(p.logits, ref_labels, -100, "mean")
    assert out.n_valid.item() == ref["n_valid"] == 18
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * ref["loss"]
    _check_grad(grad, oracle.ce_backward(p.logits, ref_labels, -100, "mean"))


def test_ignore_index_inside_vocab(lh):
    p = wl.random_ce(40, 900, torch.bfloat16, seed=10, ignore_frac=0.0)
    logits, labels = _dev(p)
    out = lh.ce_logits_fwd(logits, labels, 5, "sum")
    torch.cuda.synchronize()
    ref = oracle.ce_forward(p.logits, p.labels, 5, "sum")
    assert out.n_valid.item() == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * ref["loss"]


def test_label_in_last_column(lh):
    p = wl.random_ce(9, 1001, torch.bfloat16, seed=13, ignore_frac=0.0)
    logits, labels = _dev(p)
    labels[:] = 1000
    out = lh.ce_logits_fwd(logits, labels, -100, "sum", want_label_logit=True)
    torch.cuda.synchronize()
    assert torch.equal(out.label_logit.cpu(), p.logits[:, 1000].float())


def test_empty_batch(lh):
    logits = torch.empty(0, 128, device="cuda").bfloat16()
    labels = torch.empty(0, dtype=torch.int64, device="cuda")
    out = lh.ce_logits_fwd(logits, labels)
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and out.n_valid.item() == 0


def test_deterministic(lh):
    p = wl.random_ce(256, 20000, torch.bfloat16, seed=14)
    logits, labels = _dev(p)
    a = lh.ce_logits_fwd(logits, labels, want_rows=True)
    b = lh.ce_logits_fwd(logits, labels, want_rows=True)
    ga = lh.ce_logits_bwd(logits, labels, a.lse, a.n_valid, torch.ones(1, device="cuda"))
    gb = lh.ce_logits_bwd(logits, labels, b.lse, b.n_valid, torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a.loss, b.loss) and torch.equal(a.loss_rows, b.loss_rows)
    assert torch.equal(ga, gb)


def test_full_size_workload_against_the_full_oracle(lh):
    """[16384, 128256] bf16, 5% ignored, sum, in place: the launches the benchmark
    times.  Every row's lse, loss and gathered label logit, n_valid, the loss,
    and all 2.1e9 entries of the in-place gradient against the fp64 oracle
    (the gradient in blocks of rows, with the blockwise form of the
    specification's max-relative and normwise errors)."""
    p = wl.ce_logits_large(device="cuda")
    host = p.logits.cpu()  # the inputs, before the backward overwrites them
    labels = p.labels.cpu()
    out = lh.ce_logits_fwd(p.logits, p.labels, -100, "sum", want_rows=True,
                           want_label_logit=True)
    g = torch.ones(1, device="cuda")
    lh.ce_logits_bwd(p.logits, p.labels, out.lse, out.n_valid, g, inplace_grad=True)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    ref = oracle.ce_forward(host, labels)
    _check_fwd(out, ref)
    assert int(out.n_valid.item()) == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    # the loss is the sum of the rows: within the sum of their bounds
    assert abs(out.loss.item() - ref["loss"]) <= np.sum(2 * 5e-5 * (1 + np.abs(ref["lse"])))
    lr = out.loss_rows.cpu().double().numpy()
    assert np.all(np.abs(lr - ref["loss_rows"]) <= 2 * 5e-5 * (1 + np.abs(ref["lse"])))
    valid = labels.numpy() != -100
    zl = out.label_logit.cpu().double().numpy()
    assert np.array_equal(zl[valid], ref["label_logit"][valid])  # the bf16 value, widened
    dz = p.logits.cpu()
    del p
    acc = oracle.BlockwiseError()
    for r0 in range(0, dz.shape[0], 1024):
        rows = np.arange(r0, min(dz.shape[0], r0 + 1024))
        acc.add(dz[r0:r0 + 1024], oracle.ce_backward(host, labels, rows=rows))
    assert acc.max_rel() <= 2e-2 and acc.normwise() <= 5e-3, (acc.max_rel(), acc.normwise())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("col0", [1, 3, 8])
def test_ce_on_a_column_slice(lh, dtype, col0):
    # logits that start inside a 16-byte block: columns [col0, col0 + V) of a
    # wider buffer; in place and out of place
    N, V, W = 70, 5003, 5020
    full = wl.random_ce(N, W, dtype, seed=col0 + 40).logits
    p = wl.random_ce(N, V, dtype, seed=col0 + 41, reduction="mean")
    x_host = full[:, col0:col0 + V]
    dev_full = full.cuda()
    x = dev_full[:, col0:col0 + V]
    labels = p.labels.cuda()
    out = lh.ce_logits_fwd(x, labels, -100, "mean")
    ref = oracle.ce_forward(x_host, p.labels, -100, "mean")
    _check_fwd(out, ref)
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    g = torch.tensor([1.5], device="cuda")
    want = oracle.ce_backward(x_host, p.labels, -100, "mean", grad_loss=1.5)
    grad = lh.ce_logits_bwd(x, labels, out.lse, out.n_valid, g, -100, "mean")
    torch.cuda.synchronize()
    _check_grad(grad, want)
    before = dev_full.clone()
    lh.ce_logits_bwd(x, labels, out.lse, out.n_valid, g, -100, "mean", inplace_grad=True,
                     status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    _check_grad(x, want)
    # the columns outside the slice are untouched
    assert torch.equal(dev_full[:, :col0], before[:, :col0])
    assert torch.equal(dev_full[:, col0 + V:], before[:, col0 + V:])
