"""CE forward and backward in one call (ce_logits_fwd_bwd) vs the fp64 oracle.

Rows that fit a cluster are read once: the row-cluster kernel forms each
row's lse, its loss and its gradient; longer rows, and a gradient buffer whose
rows sit at other offsets within their 16-byte blocks than the logits rows,
run the forward and the backward.  The cases reach clusters of 1, 2, 4 and 8
CTAs, rows that start and end inside a block, the twice-streamed long rows
and the register-streaming row kernel.  Bars, as for the separate calls:
loss 1e-3 relative, lse 5e-5 (1 + |lse|) on rows with a valid label, n_valid
exact, gradient max relative 2e-2 and normwise 5e-3.  Against the separate
forward and backward of the same inputs the loss agrees to 1e-5 relative and
the gradient to one rounding flip per element (the lse is summed in another
order: a few fp32 ulp).
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


def _check_grad(got, want):
    assert oracle.max_rel_err(got.float().cpu(), want) <= 2e-2
    assert oracle.normwise_err(got.float().cpu(), want) <= 5e-3


def _close(a, b, dtype, c):
    # c: the row scale; c * 2^-20 absorbs the cancellation residue of the label
    # entry c * (p_y - 1) when p_y is near 1
    rel = 1e-2 if dtype == torch.bfloat16 else 1e-5
    a, b = a.float(), b.float()
    assert torch.all((a - b).abs() <= rel * b.abs() + abs(c) * 2.0**-20), \
        (a - b).abs().max().item()


CASES = [
    # dtype, N, V, ld                          path
    (torch.bfloat16, 300, 1000, 1000),       # cluster of 1
    (torch.float32, 130, 4100, 4104),        # cluster of 1, padded row stride
    (torch.bfloat16, 700, 50264, 50264),     # cluster of 2
    (torch.bfloat16, 300, 120008, 120008),   # cluster of 4, last slice shorter
    (torch.bfloat16, 40, 128256, 128256),    # cluster of 4, the Llama-3 vocabulary
    (torch.float32, 100, 128256, 128256),    # cluster of 8
    (torch.bfloat16, 6, 300000, 300000),     # too long for a cluster: forward, then backward
    (torch.bfloat16, 77, 1003, 1011),        # rows inside 16-byte blocks, cluster of 1
    (torch.bfloat16, 120, 50257, 50257),     # GPT-2 vocabulary: rows inside blocks, cluster of 2
    (torch.float32, 30, 32777, 32777),       # rows inside blocks, cluster of 4
]


@pytest.mark.parametrize("dtype,N,V,ld", CASES)
@pytest.mark.parametrize("reduction,nlt,g", [("sum", None, None), ("mean", None, 1.3),
                                             ("sum", 5000, 0.7)])
def test_fwd_bwd_parity(lh, dtype, N, V, ld, reduction, nlt, g):
    p = wl.random_ce(N, V, dtype, seed=N + V + 3, ignore_frac=0.1, reduction=reduction,
                     num_label_tokens=nlt, ld=ld)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    gl = None if g is None else torch.tensor([g], device="cuda")
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, reduction, nlt, gl, want_lse=True)
    sep = lh.ce_logits_fwd(logits, labels, -100, reduction, nlt)
    sep_grad = lh.ce_logits_bwd(logits, labels, sep.lse, sep.n_valid,
                                torch.tensor([1.0 if g is None else g], device="cuda"), -100,
                                reduction, nlt)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    ref = oracle.ce_forward(p.logits, p.labels, -100, reduction, nlt)
    assert out.n_valid.item() == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    valid = (p.labels != -100).numpy()
    lse = out.lse.cpu().double().numpy()[valid]
    want = ref["lse"][valid]
    assert np.all(np.abs(lse - want) <= 5e-5 * (1 + np.abs(want)))
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, reduction, nlt,
                                         grad_loss=1.0 if g is None else g))
    assert abs(out.loss.item() - sep.loss.item()) <= 1e-5 * abs(sep.loss.item())
    div = nlt if nlt is not None else (ref["n_valid"] if reduction == "mean" else 1)
    _close(grad, sep_grad, dtype, (1.0 if g is None else g) / max(div, 1))
    assert torch.count_nonzero(grad.cpu()[torch.from_numpy(~valid)]) == 0


@pytest.mark.parametrize("dtype,N,V", [(torch.bfloat16, 100, 128256), (torch.float32, 64, 50264),
                                       (torch.bfloat16, 33, 1003)])
def test_fwd_bwd_inplace(lh, dtype, N, V):
    p = wl.random_ce(N, V, dtype, seed=V + 2)
    logits, labels = p.logits.cuda().contiguous(), p.labels.cuda()
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, "mean", inplace_grad=True)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert grad.data_ptr() == logits.data_ptr()
    ref = oracle.ce_forward(p.logits, p.labels, -100, "mean")
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, "mean"))


def test_fwd_bwd_out_of_range_labels(lh):
    # aligned rows (the one-pass kernel): bad labels set the status and count as ignored
    p = wl.random_ce(64, 4096, torch.bfloat16, seed=21, ignore_frac=0.0)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    labels[3] = 4096
    labels[9] = -7
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, "mean")
    torch.cuda.synchronize()
    assert int(out.status.item()) == -5
    ref_labels = p.labels.clone()
    ref_labels[3] = -100
    ref_labels[9] = -100
    ref = oracle.ce_forward(p.logits, ref_labels, -100, "mean")
    assert out.n_valid.item() == ref["n_valid"] == 62
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    _check_grad(grad, oracle.ce_backward(p.logits, ref_labels, -100, "mean"))


@pytest.mark.parametrize("V", [4096, 1003])
def test_fwd_bwd_degenerate(lh, V):
    # all rows ignored; num_label_tokens = 0; one valid row
    p = wl.random_ce(50, V, torch.bfloat16, seed=V)
    logits = p.logits.cuda()
    none = torch.full((50,), -100, dtype=torch.int64, device="cuda")
    out, grad = lh.ce_logits_fwd_bwd(logits, none, -100, "mean")
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and out.n_valid.item() == 0
    assert torch.count_nonzero(grad) == 0
    labels = p.labels.cuda()
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, "sum", 0)
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and torch.count_nonzero(grad) == 0
    one = none.clone()
    one[17] = 5
    out, grad = lh.ce_logits_fwd_bwd(logits, one, -100, "mean")
    torch.cuda.synchronize()
    lh.check_status(out.status)
    ref_labels = torch.full((50,), -100, dtype=torch.int64)
    ref_labels[17] = 5
    ref = oracle.ce_forward(p.logits, ref_labels, -100, "mean")
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    _check_grad(grad, oracle.ce_backward(p.logits, ref_labels, -100, "mean"))


def test_fwd_bwd_empty(lh):
    logits = torch.zeros((0, 4096), dtype=torch.bfloat16, device="cuda")
    labels = torch.zeros(0, dtype=torch.int64, device="cuda")
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, "mean")
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and out.n_valid.item() == 0 and grad.shape == (0, 4096)


def test_fwd_bwd_deterministic(lh):
    p = wl.random_ce(500, 128256, torch.bfloat16, seed=13)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    a, ga = lh.ce_logits_fwd_bwd(logits, labels, -100, "sum", want_lse=True)
    b, gb = lh.ce_logits_fwd_bwd(logits, labels, -100, "sum", want_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(a.loss, b.loss) and torch.equal(ga, gb)
    assert torch.equal(a.lse.nan_to_num(0.0), b.lse.nan_to_num(0.0))  # NaN: rows not read


def test_fwd_bwd_rejects_bad_buffers(lh):
    from lm_head_linear_fwd_gb300 import _abi
    N, V = 8, 64
    logits = torch.zeros((N, V), dtype=torch.bfloat16, device="cuda")
    labels = torch.zeros(N, dtype=torch.int64, device="cuda")
    loss = torch.zeros(1, device="cuda")
    nv = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(_abi.ce_logits_fwd_bwd_workspace_bytes(N, V), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(grad_ptr, ld_grad, inplace, ws_bytes):
        return _abi.ce_logits_fwd_bwd(logits.data_ptr(), _abi.FLCE_BF16, N, V, V,
                                      labels.data_ptr(), -100, _abi.FLCE_SUM, -1, None,
                                      loss.data_ptr(), nv.data_ptr(), None, inplace, grad_ptr,
                                      ld_grad, ws.data_ptr(), ws_bytes, st.data_ptr(), s)

    other = torch.empty_like(logits)
    assert call(other.data_ptr(), V, 0, ws.numel()) == 0
    assert call(logits.data_ptr() + 2 * V, V, 0, ws.numel()) == -1  # overlaps the logits
    assert call(other.data_ptr(), V, 1, ws.numel()) == -1           # in place, elsewhere
    assert call(other.data_ptr(), V - 1, 0, ws.numel()) == -2       # ld_grad < V
    assert call(other.data_ptr(), V, 0, ws.numel() - 1) == -6       # workspace too small
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("inplace", [False, True])
def test_eager_autograd(lh, inplace):
    p = wl.random_ce(257, 50264, torch.bfloat16, seed=17)
    labels = p.labels.cuda()
    grads, losses = [], []
    for eager in (False, True):
        x = p.logits.cuda().requires_grad_(True)
        loss = lh.ce_logits(x, labels, reduction="mean", eager=eager,
                            inplace_grad=inplace and eager)
        (2.0 * loss).backward()
        grads.append(x.grad)
        losses.append(loss.detach())
    torch.cuda.synchronize()
    assert abs(losses[1].item() - losses[0].item()) <= 1e-5 * abs(losses[0].item())
    _close(grads[1], grads[0], torch.bfloat16, 2.0 / int((p.labels != -100).sum()))
    _check_grad(grads[1], oracle.ce_backward(p.logits, p.labels, -100, "mean", grad_loss=2.0))


def test_eager_second_backward_raises(lh):
    p = wl.random_ce(16, 1024, torch.bfloat16, seed=3)
    x = p.logits.cuda().requires_grad_(True)
    loss = lh.ce_logits(x, p.labels.cuda(), eager=True)
    loss.backward(retain_graph=True)
    with pytest.raises(RuntimeError):
        loss.backward()


def test_fwd_bwd_full_size_sampled(lh):
    """[16384, 128256] bf16, 5% ignored, sum, in place: sampled rows against the
    oracle one by one, the loss against the fp64 sum of the per-row losses of
    the separate forward."""
    p = wl.ce_logits_large(device="cuda")
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(p.N, 48, replace=False))
    host_rows = p.logits[rows].cpu()
    host_labels = p.labels[rows].cpu()
    sep = lh.ce_logits_fwd(p.logits, p.labels, -100, "sum", want_rows=True)
    out, _ = lh.ce_logits_fwd_bwd(p.logits, p.labels, -100, "sum", inplace_grad=True,
                                  want_lse=True)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    ref = oracle.ce_forward(host_rows, host_labels)
    valid = (host_labels != -100).numpy()
    lse = out.lse.cpu().double().numpy()[rows][valid]
    assert np.all(np.abs(lse - ref["lse"][valid]) <= 5e-5 * (1 + np.abs(ref["lse"][valid])))
    lr = sep.loss_rows.cpu().double().numpy()
    assert abs(out.loss.item() - lr.sum()) <= 1e-5 * abs(lr.sum())
    assert out.n_valid.item() == int((p.labels != -100).sum())
    _check_grad(p.logits[rows].cpu(), oracle.ce_backward(host_rows, host_labels))


@pytest.mark.parametrize("col0", [1, 8])
def test_fwd_bwd_column_slice_in_place(lh, col0):
    # a column slice that starts inside a 16-byte block, its gradient written
    # in place: the neighbouring columns are untouched
    N, V, W = 64, 5003, 5024
    full = wl.random_ce(N, W, torch.bfloat16, seed=col0 + 60).logits
    labels = wl.random_ce(N, V, torch.bfloat16, seed=col0 + 61).labels
    x_host = full[:, col0:col0 + V]
    dev_full = full.cuda()
    before = dev_full.clone()
    x = dev_full[:, col0:col0 + V]
    out, grad = lh.ce_logits_fwd_bwd(x, labels.cuda(), -100, "sum", inplace_grad=True)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    ref = oracle.ce_forward(x_host, labels, -100, "sum")
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    _check_grad(x, oracle.ce_backward(x_host, labels, -100, "sum"))
    assert torch.equal(dev_full[:, :col0], before[:, :col0])
    assert torch.equal(dev_full[:, col0 + V:], before[:, col0 + V:])


def test_fwd_bwd_grad_rows_at_other_offsets(lh):
    # gradient rows at other offsets within their blocks: forward, then the
    # register-streaming backward
    N, V = 50, 3001
    p = wl.random_ce(N, V, torch.bfloat16, seed=66, reduction="mean")
    logits, labels = p.logits.cuda().contiguous(), p.labels.cuda()
    big = torch.full((N * V + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    gbuf = big[3:3 + N * V].view(N, V)
    out, grad = lh.ce_logits_fwd_bwd(logits, labels, -100, "mean", grad_logits=gbuf)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert torch.all(torch.isnan(big[:3])) and torch.all(torch.isnan(big[3 + N * V:]))
    ref = oracle.ce_forward(p.logits, p.labels, -100, "mean")
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, "mean"))
