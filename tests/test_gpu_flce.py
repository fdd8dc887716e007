"""Fused linear cross-entropy: CUDA path through the C ABI vs the fp64 oracle.

Tolerances (derived in tests/tolerances.py):
* loss: |gpu - ref| <= 1e-3 |ref|;
* per-row lse: |gpu - ref| <= 2e-5 (1 + |ref|) for bf16 inputs (fp32
  accumulation of exact bf16 products; a lost 256-column vocabulary tile moves
  lse by ~2e-3 at V = 128256, 7x over); for fp32 inputs the fp64 effect of the
  tf32 operand cut plus that bound; per-row loss twice the lse bound;
* n_valid exact;
* grad_H, grad_W, grad_b: max relative <= 2e-2, normwise <= 5e-3 (dZ is rounded
  to the input dtype before the two gradient contractions).
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
    tol.check_grad(got.float().cpu(), want, name, oracle)


def _run(lh, p, chunk=None, g=1.0, accumulate_init=None):
    H, W, b, y = _to(p)
    out = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, want_rows=True,
                      want_label_logit=True)
    gw = None
    if accumulate_init is not None:
        gw = accumulate_init.cuda().clone()
    bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.tensor([g], device="cuda"), b, -100,
                     p.reduction, p.num_label_tokens, chunk, grad_W=gw,
                     accumulate_grad_W=accumulate_init is not None, status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    return out, bw


def _check_all(p, out, bw, g=1.0, grad_W_init=None, W64=None):
    W = p.W if W64 is None else W64
    ref = oracle.flce_forward(p.H, W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens)
    assert int(out.n_valid.item()) == ref["n_valid"]
    tol.check_loss(out.loss.item(), ref["loss"])
    tol.check_flce_lse(out.lse, ref["lse"], p.H, W, p.bias)
    if out.loss_rows is not None:
        tol.check_flce_loss_rows(out.loss_rows, ref["loss_rows"], ref["lse"], p.H, W)
    gr = oracle.flce_backward(p.H, W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens,
                              grad_loss=g, grad_W_init=grad_W_init)
    _grad_ok(bw.grad_H, gr["grad_H"], "grad_H")
    _grad_ok(bw.grad_W, gr["grad_W"], "grad_W")
    if p.bias is not None:
        _grad_ok(bw.grad_bias, gr["grad_b"], "grad_b")


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_tiny_fp32_workload(lh, reduction):
    """N=256, D=128, V=1000, fp32 (tf32 tensor cores), 10% ignored."""
    p = wl.tiny_flce(reduction)
    out, bw = _run(lh, p, g=1.5)
    _check_all(p, out, bw, g=1.5)


def test_small_model_workload(lh):
    """B=2, T=1024, D=768, V=32777 (odd), bf16 with bias, mean."""
    p = wl.small_flce()
    out, bw = _run(lh, p)
    _check_all(p, out, bw)


@pytest.mark.parametrize("pair", [31, 0, 32], ids=["pair", "single", "wide_dz"])
@pytest.mark.parametrize("N,D,V,chunk,bias", [(700, 256, 3001, 256, True), (129, 64, 777, 128, False),
                                              (1000, 520, 2048, None, False)])
def test_ragged_multi_chunk(lh, N, D, V, chunk, bias, pair):
    from lm_head_linear_fwd_gb300 import _abi
    prev = _abi.flce_gemm_set_pair(pair)
    try:
        p = wl.random_flce(N, D, V, torch.bfloat16, bias=bias, seed=N, reduction="mean")
        out, bw = _run(lh, p, chunk=chunk, g=0.5)
        _check_all(p, out, bw, g=0.5)
    finally:
        _abi.flce_gemm_set_pair(prev)


def test_fp32_multi_chunk_with_bias(lh):
    p = wl.random_flce(300, 96, 1234, torch.float32, bias=True, seed=31, reduction="sum",
                       num_label_tokens=250)
    out, bw = _run(lh, p, chunk=128)
    _check_all(p, out, bw)


def test_accumulate_grad_W(lh):
    p = wl.random_flce(256, 128, 1000, torch.bfloat16, seed=41)
    init = torch.randn(1000, 128) * 0.01
    out, bw = _run(lh, p, accumulate_init=init)
    _check_all(p, out, bw, grad_W_init=init.double().numpy())


def test_label_logit_and_rows(lh):
    p = wl.random_flce(200, 64, 1000, torch.bfloat16, seed=51)
    p.labels[:5] = 999   # label in the last (partial) vocabulary tile
    p.labels[5:9] = 0
    out, _ = _run(lh, p)
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, "sum")
    zl = out.label_logit.cpu().double().numpy()
    v = p.labels.numpy() != -100
    # the label logit carries the accumulation error of one logit (the lse bound)
    assert np.all(np.abs(zl[v] - ref["label_logit"][v]) <=
                  tol.flce_lse_bound_bf16(ref["label_logit"][v]))
    assert np.all(np.isnan(zl[~v]))
    lr = out.loss_rows.cpu().double().numpy()
    assert np.all(lr[~v] == 0) and np.all(lr >= -1e-4)


@pytest.mark.parametrize("reduction,nlt", [("mean", None), ("sum", 0)])
def test_zero_guards(lh, reduction, nlt):
    p = wl.random_flce(150, 64, 500, torch.bfloat16, bias=True, seed=61, reduction=reduction,
                       num_label_tokens=nlt)
    if nlt is None:
        p.labels[:] = -100
    out, bw = _run(lh, p)
    assert out.loss.item() == 0.0
    for t in (bw.grad_H, bw.grad_W, bw.grad_bias):
        assert torch.count_nonzero(t).item() == 0


def test_bad_label_status(lh):
    p = wl.random_flce(64, 64, 300, torch.bfloat16, seed=71, ignore_frac=0.0)
    H, W, b, y = _to(p)
    y[10] = 300
    out = lh.flce_fwd(H, W, y, b)
    torch.cuda.synchronize()
    assert int(out.status.item()) == -5
    assert out.n_valid.item() == 63


def test_autograd_module(lh):
    p = wl.random_flce(300, 128, 2000, torch.bfloat16, bias=True, seed=81, reduction="mean")
    H, W, b, y = _to(p)
    for t in (H, W, b):
        t.requires_grad_(True)
    loss = lh.flce(H, W, y, b, reduction="mean", chunk=128)
    loss.backward()
    torch.cuda.synchronize()
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, "mean")
    _grad_ok(H.grad, gr["grad_H"], "grad_H")
    _grad_ok(W.grad, gr["grad_W"], "grad_W")
    _grad_ok(b.grad, gr["grad_b"], "grad_b")
    with pytest.raises(RuntimeError):
        (gH,) = torch.autograd.grad(lh.flce(H, W, y, b), H, create_graph=True)
        gH.sum().backward()


def test_mask_argument(lh):
    p = wl.random_flce(128, 64, 400, torch.bfloat16, seed=91, ignore_frac=0.0)
    H, W, b, y = _to(p)
    mask = torch.ones(128, dtype=torch.int64, device="cuda")
    mask[::3] = 0
    loss = lh.flce(H, W, y, None, mask=mask, reduction="sum")
    labels = p.labels.clone()
    labels[::3] = -100
    ref = oracle.flce_forward(p.H, p.W, None, labels, -100, "sum")
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * ref["loss"]


def test_deterministic(lh):
    p = wl.random_flce(600, 256, 5000, torch.bfloat16, bias=True, seed=101)
    o1, b1 = _run(lh, p, chunk=256)
    o2, b2 = _run(lh, p, chunk=256)
    assert torch.equal(o1.loss, o2.loss) and torch.equal(o1.lse, o2.lse)
    for a, c in ((b1.grad_H, b2.grad_H), (b1.grad_W, b2.grad_W), (b1.grad_bias, b2.grad_bias)):
        assert torch.equal(a, c)


def _sampled_full_size(lh, p, n_rows=32, sub_rows=256):
    """Full-size run (the benchmark's launches) of a problem too large for the
    host oracle as a whole, checked on sampled rows and by the row-linearity
    of grad_W; the complete gradients are then checked on a row subset run as
    its own problem."""
    H, W, b, y = _to(p)
    out = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, want_rows=True)
    one = torch.ones(1, device="cuda")
    bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, one, b, -100, p.reduction,
                     p.num_label_tokens)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    nv = int((p.labels != -100).sum())
    assert out.n_valid.item() == nv
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(p.N, n_rows, replace=False))
    Hc, yc = p.H.cpu(), p.labels.cpu()
    W64 = p.W.cpu().double().numpy()  # widened once, reused by every oracle call
    ref = oracle.flce_forward(Hc, W64, None, yc, -100, p.reduction, p.num_label_tokens, rows=rows)
    lse = out.lse.cpu().double().numpy()[rows]
    tol.check_flce_lse(lse, ref["lse"], Hc, W64)
    lr = out.loss_rows.cpu().double().numpy()
    tol.check_flce_loss_rows(lr[rows], ref["loss_rows"], ref["lse"], Hc, W64)
    total = lr.sum() / (p.num_label_tokens if p.num_label_tokens else 1)
    assert abs(out.loss.item() - total) <= 1e-5 * abs(total)
    gr = oracle.flce_backward(Hc, W64, None, yc, -100, p.reduction, p.num_label_tokens, rows=rows,
                              n_valid_total=nv, want_grad_W=False)
    _grad_ok(bw.grad_H[torch.as_tensor(rows, device="cuda")], gr["grad_H"], "grad_H rows")
    # grad_W is linear in the rows: a full run equals two half runs accumulated
    half = (p.N // 2) // 128 * 128
    gW2 = torch.zeros_like(bw.grad_W)
    for r0, r1, acc in ((0, half, False), (half, p.N, True)):
        lh.flce_bwd(H[r0:r1], W, y[r0:r1], out.lse[r0:r1], out.n_valid, one, None, -100,
                    p.reduction, p.num_label_tokens, want_grad_H=False, grad_W=gW2,
                    accumulate_grad_W=acc)
    torch.cuda.synchronize()
    assert oracle.normwise_err(gW2.cpu(), bw.grad_W.cpu().double().numpy()) <= 1e-5
    # complete gradients of a row subset, as a problem of its own
    sub = torch.as_tensor(np.sort(rng.choice(p.N, sub_rows, replace=False)))
    q = wl.FLCEInputs("subset", Hc[sub].contiguous(), p.W, None, yc[sub].contiguous(), -100,
                      p.reduction, None)
    out_s, bw_s = _run(lh, q)
    _check_all(q, out_s, bw_s, W64=W64)


def test_llama3_8b_workload_against_the_full_oracle(lh):
    """N=8192, D=4096, V=128256 bf16, Zipf labels, 3% ignored, sum / num_label_tokens,
    in the launch configuration the benchmark times (default chunk): every row's
    lse and loss, the loss, and all of grad_H and grad_W against the fp64 oracle
    over the whole problem (8NDV = 3.4e13 fp64 flops on the host cores, one to
    two minutes).  grad_W is also checked by its row-linearity (a full run
    equals two half runs accumulated)."""
    p = wl.llama3_8b_flce(device="cuda")
    H, W, b, y = _to(p)
    out = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, want_rows=True)
    one = torch.ones(1, device="cuda")
    bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, one, b, -100, p.reduction,
                     p.num_label_tokens)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    gH, gW = bw.grad_H.cpu(), bw.grad_W.cpu()
    lse, rows, loss = out.lse.cpu(), out.loss_rows.cpu(), out.loss.item()
    # row-linearity of grad_W on the device, before the host copies are compared
    half = (p.N // 2) // 128 * 128
    gW2 = torch.zeros_like(bw.grad_W)
    for r0, r1, acc in ((0, half, False), (half, p.N, True)):
        lh.flce_bwd(H[r0:r1], W, y[r0:r1], out.lse[r0:r1], out.n_valid, one, None, -100,
                    p.reduction, p.num_label_tokens, want_grad_H=False, grad_W=gW2,
                    accumulate_grad_W=acc)
    torch.cuda.synchronize()
    assert oracle.normwise_err(gW2.cpu(), gW.double().numpy()) <= 1e-5
    nv = int(out.n_valid.item())
    Hc, yc, Wc = p.H.cpu(), p.labels.cpu(), p.W.cpu()
    del H, W, y, bw, out, gW2, p
    torch.cuda.empty_cache()
    W64 = Wc.double().numpy()
    del Wc
    gr = oracle.flce_backward(Hc, W64, None, yc, -100, "sum", nv, with_forward=True)
    ref = gr["forward"]
    assert nv == ref["n_valid"]
    tol.check_loss(loss, ref["loss"])
    tol.check_flce_lse(lse, ref["lse"], Hc, W64)
    tol.check_flce_loss_rows(rows, ref["loss_rows"], ref["lse"], Hc, W64)
    # the loss is the sum of the rows: within the sum of their bounds
    row_bound = 2.0 * tol.flce_lse_bound_bf16(ref["lse"])
    assert abs(loss - ref["loss"]) <= row_bound[ref["loss_rows"] != 0].sum() / nv
    _grad_ok(gH, gr["grad_H"], "grad_H")
    del gr["grad_H"]
    _grad_ok(gW, gr["grad_W"], "grad_W")


def test_long_packed_workload_sampled(lh):
    """N=65536 (4 x 16384 packed), D=5120, V=151936 bf16, ~8% ignored, sum."""
    p = wl.long_packed_flce(device="cuda")
    _sampled_full_size(lh, p, n_rows=16, sub_rows=128)


@pytest.mark.parametrize("pair", [31, 0, 32], ids=["pair", "single", "wide_dz"])
@pytest.mark.parametrize("N,D,V,vslice,bias,reduction", [
    (700, 256, 3001, 1024, True, "mean"),    # three slices, the last 953 columns
    (1000, 520, 2048, 256, False, "sum"),    # eight slices of one tile each
    (129, 64, 777, 512, True, "sum"),        # a ragged row tile and a ragged slice
    (300, 128, 20000, 20224, False, "mean"),  # one slice wider than V
])
def test_vocabulary_slices(lh, N, D, V, vslice, bias, reduction, pair):
    """The backward split over vocabulary slices (chunk = -columns): all rows
    per slice, grad_W written slice by slice, grad_H accumulated in fp32 and
    rounded once, bias columns per slice."""
    from lm_head_linear_fwd_gb300 import _abi
    prev = _abi.flce_gemm_set_pair(pair)
    try:
        p = wl.random_flce(N, D, V, torch.bfloat16, bias=bias, seed=N + 7, reduction=reduction)
        out, bw = _run(lh, p, chunk=-vslice, g=0.75)
        _check_all(p, out, bw, g=0.75)
    finally:
        _abi.flce_gemm_set_pair(prev)


def test_vocabulary_slices_accumulate_grad_W(lh):
    p = wl.random_flce(256, 128, 1000, torch.bfloat16, seed=43)
    init = torch.randn(1000, 128) * 0.01
    out, bw = _run(lh, p, chunk=-256, accumulate_init=init)
    _check_all(p, out, bw, grad_W_init=init.double().numpy())


def test_vocabulary_slices_match_row_chunks(lh):
    """Both splits of the same backward: the same dZ values feed the same
    contractions, in another order of fp32 additions for grad_H (slices) and
    grad_W (chunks): the gradients agree to fp32 summation order plus one bf16
    rounding of grad_H."""
    p = wl.random_flce(1536, 256, 6000, torch.bfloat16, bias=True, seed=5, reduction="mean")
    H, W, b, y = _to(p)
    out = lh.flce_fwd(H, W, y, b, -100, "mean")
    g = torch.ones(1, device="cuda")
    rows = lh.flce_bwd(H, W, y, out.lse, out.n_valid, g, b, -100, "mean", None, 512)
    sl = lh.flce_bwd(H, W, y, out.lse, out.n_valid, g, b, -100, "mean", None, -1536)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    # fp32 sums of 1536 products in another order (one tensor-core sweep
    # against three of 512 added in L2): ~1e-6, the bound of the row-linearity
    # checks
    assert oracle.normwise_err(sl.grad_W.cpu(), rows.grad_W.cpu().double().numpy()) <= 1e-5
    assert oracle.normwise_err(sl.grad_bias.cpu(), rows.grad_bias.cpu().double().numpy()) <= 1e-5
    assert oracle.normwise_err(sl.grad_H.float().cpu(),
                               rows.grad_H.float().cpu().double().numpy()) <= 4e-3


def test_vocabulary_slices_rejected_for_fp32(lh):
    p = wl.random_flce(64, 64, 300, torch.float32, seed=8)
    H, W, b, y = _to(p)
    out = lh.flce_fwd(H, W, y, b)
    with pytest.raises(lh.FlceError):
        lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b, -100, "sum",
                    None, -256)


@pytest.mark.parametrize("pair", [58, 31], ids=["default", "no_wide_dz"])
@pytest.mark.parametrize("chunk", [None, 128], ids=["one_chunk", "three_chunks"])
@pytest.mark.parametrize("want", [(True, True, True), (False, True, True), (True, False, True),
                                  (False, False, True), (True, True, False)],
                         ids=["all", "no_H", "no_W", "bias_only", "no_bias"])
def test_gradient_subsets_with_split_k(lh, want, chunk, pair):
    """Every subset of the gradients at a shape whose grad_H is split over K
    (three 128-row tiles, V = 5000): the bias column sums and the split-K close
    are done by the epilogue warps of whichever contraction follows, or by
    kernels of their own when none does; each requested gradient against the
    oracle, whatever the others."""
    from lm_head_linear_fwd_gb300 import _abi
    want_h, want_w, want_b = want
    prev = _abi.flce_gemm_set_pair(pair)
    try:
        p = wl.random_flce(300, 256, 5000, torch.bfloat16, bias=True, seed=303, reduction="mean")
        H, W, b, y = _to(p)
        out = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens)
        bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.tensor([0.75], device="cuda"), b,
                         -100, p.reduction, p.num_label_tokens, chunk, want_grad_H=want_h,
                         want_grad_W=want_w, want_grad_bias=want_b, status=out.status)
        torch.cuda.synchronize()
        lh.check_status(out.status)
        gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, p.reduction,
                                  p.num_label_tokens, grad_loss=0.75)
        assert (bw.grad_H is not None) == want_h and (bw.grad_W is not None) == want_w
        assert (bw.grad_bias is not None) == want_b
        if want_h:
            _grad_ok(bw.grad_H, gr["grad_H"], "grad_H")
        if want_w:
            _grad_ok(bw.grad_W, gr["grad_W"], "grad_W")
        if want_b:
            _grad_ok(bw.grad_bias, gr["grad_b"], "grad_b")
    finally:
        _abi.flce_gemm_set_pair(prev)
