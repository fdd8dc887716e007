"""CE backward on given logits with no saved lse (lse = NULL through the C ABI).

The backward then forms each row's lse again before the gradient.  Three
kernels serve it, chosen by the row's length and alignment:
* rows of at most 8 x 64 KiB: a thread-block cluster of P = 1, 2, 4 or 8 CTAs
  holds the row's 16-byte blocks in shared memory (the cases below reach every
  P, slices of unequal length, more rows than resident clusters, and rows that
  start and end inside a block, whose first and last blocks are finished
  element by element);
* longer rows: the bulk-copy ring, streaming each row twice;
* a gradient buffer whose rows start at other offsets within a 16-byte block
  than the logits rows: the register-streaming row kernel.

Each case is checked against the fp64 oracle with the gradient bars of the
other CE tests (max relative 2e-2, normwise 5e-3) and against the saved-lse
backward of the same inputs: both round the same softmax once to the output
dtype, and the recomputed lse differs from the saved one by a few fp32 ulp
(about 1e-6 relative in each softmax entry), so the two differ by at most one
rounding flip per element: 2^-7 relative for bf16 (bound 1e-2), and for fp32
about 1e-6 (bound 1e-5).
"""
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


def _close_to_saved(a, b, dtype, c):
    # c: the row scale g * scale.  The label entry c * (p_y - 1) cancels when
    # p_y is near 1 (V = 1 gives exactly 0 in exact arithmetic): there both
    # kernels leave a residue of a few fp32 ulp of c, hence the floor c * 2^-20.
    rel = 1e-2 if dtype == torch.bfloat16 else 1e-5
    a, b = a.float(), b.float()
    assert torch.all((a - b).abs() <= rel * b.abs() + abs(c) * 2.0**-20), \
        (a - b).abs().max().item()


CASES = [
    # dtype, N, V, ld                          path (CTAs per row)
    (torch.bfloat16, 300, 1000, 1000),       # cluster of 1
    (torch.float32, 130, 4100, 4104),        # cluster of 1, padded row stride
    (torch.bfloat16, 200, 32768, 32768),     # cluster of 1, a slice of exactly 64 KiB
    (torch.bfloat16, 700, 50264, 50264),     # cluster of 2, slices 3142 / 3141 vectors
    (torch.bfloat16, 300, 120008, 120008),   # cluster of 4, last slice shorter
    (torch.bfloat16, 40, 128256, 128256),    # cluster of 4, the Llama-3 vocabulary
    (torch.float32, 100, 128256, 128256),    # cluster of 8
    (torch.bfloat16, 6, 300000, 300000),     # too long for a cluster: streamed twice
    (torch.bfloat16, 77, 1003, 1011),        # rows inside 16-byte blocks, cluster of 1
    (torch.float32, 5, 32777, 32777),        # rows inside blocks, cluster of 4
    (torch.bfloat16, 200, 50257, 50257),     # GPT-2 vocabulary: rows inside blocks, cluster of 2
    (torch.bfloat16, 96, 128255, 128255),    # rows inside blocks, cluster of 4
    (torch.bfloat16, 33, 7, 7),              # rows shorter than a block
]


@pytest.mark.parametrize("dtype,N,V,ld", CASES)
@pytest.mark.parametrize("reduction,nlt", [("sum", None), ("mean", None), ("sum", 5000)])
def test_no_lse_parity(lh, dtype, N, V, ld, reduction, nlt):
    p = wl.random_ce(N, V, dtype, seed=N + V + 7, ignore_frac=0.1, reduction=reduction,
                     num_label_tokens=nlt, ld=ld)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    out = lh.ce_logits_fwd(logits, labels, -100, reduction, nlt)
    g = torch.tensor([1.3], device="cuda")
    grad = lh.ce_logits_bwd(logits, labels, None, out.n_valid, g, -100, reduction, nlt,
                            status=out.status)
    saved = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, g, -100, reduction, nlt)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, reduction, nlt,
                                         grad_loss=1.3))
    div = nlt if nlt is not None else (int(out.n_valid.item()) if reduction == "mean" else 1)
    _close_to_saved(grad, saved, dtype, 1.3 / max(div, 1))
    ignored = (p.labels == -100).numpy()
    assert torch.count_nonzero(grad.cpu()[torch.from_numpy(ignored)]) == 0


@pytest.mark.parametrize("dtype,N,V", [(torch.bfloat16, 100, 128256), (torch.float32, 64, 50264),
                                       (torch.bfloat16, 33, 1003)])
def test_no_lse_inplace(lh, dtype, N, V):
    p = wl.random_ce(N, V, dtype, seed=V + 1)
    logits, labels = p.logits.cuda().contiguous(), p.labels.cuda()
    out = lh.ce_logits_fwd(logits, labels, -100, "mean")
    g = torch.tensor([1.0], device="cuda")
    grad = lh.ce_logits_bwd(logits, labels, None, out.n_valid, g, -100, "mean",
                            inplace_grad=True, status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert grad.data_ptr() == logits.data_ptr()
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, "mean", grad_loss=1.0))


def test_no_lse_autograd_matches_saved(lh):
    p = wl.random_ce(257, 50264, torch.bfloat16, seed=11)
    labels = p.labels.cuda()
    grads = []
    for save_lse in (True, False):
        x = p.logits.cuda().requires_grad_(True)
        loss = lh.ce_logits(x, labels, reduction="mean", save_lse=save_lse)
        (2.0 * loss).backward()
        grads.append(x.grad)
    torch.cuda.synchronize()
    _close_to_saved(grads[1], grads[0], torch.bfloat16, 2.0 / int((p.labels != -100).sum()))
    _check_grad(grads[1], oracle.ce_backward(p.logits, p.labels, -100, "mean", grad_loss=2.0))


def test_no_lse_zero_rows_without_reading(lh):
    # every row ignored, and a zero incoming gradient: the output is all zeros
    p = wl.random_ce(64, 128256, torch.bfloat16, seed=5)
    logits = p.logits.cuda()
    labels = torch.full((64,), -100, dtype=torch.int64, device="cuda")
    out = lh.ce_logits_fwd(logits, labels, -100, "sum")
    grad = lh.ce_logits_bwd(logits, labels, None, out.n_valid, torch.ones(1, device="cuda"),
                            -100, "sum")
    assert torch.count_nonzero(grad) == 0
    labels2 = p.labels.cuda()
    out2 = lh.ce_logits_fwd(logits, labels2, -100, "sum")
    grad2 = lh.ce_logits_bwd(logits, labels2, None, out2.n_valid, torch.zeros(1, device="cuda"),
                             -100, "sum")
    torch.cuda.synchronize()
    assert torch.count_nonzero(grad2) == 0


def test_no_lse_deterministic(lh):
    p = wl.random_ce(500, 128256, torch.bfloat16, seed=9)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    out = lh.ce_logits_fwd(logits, labels, -100, "sum")
    g = torch.ones(1, device="cuda")
    a = lh.ce_logits_bwd(logits, labels, None, out.n_valid, g)
    b = lh.ce_logits_bwd(logits, labels, None, out.n_valid, g)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_no_lse_rejected_for_a_shard(lh):
    from lm_head_linear_fwd_gb300 import _abi
    logits = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    labels = torch.zeros(4, dtype=torch.int64, device="cuda")
    nv = torch.ones(1, dtype=torch.int64, device="cuda")
    g = torch.ones(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(logits)
    rc = _abi.ce_logits_bwd_shard(logits.data_ptr(), _abi.FLCE_BF16, 4, 64, 64, 0, 128,
                                  labels.data_ptr(), -100, _abi.FLCE_SUM, -1, None,
                                  nv.data_ptr(), g.data_ptr(), 0, out.data_ptr(), 64,
                                  st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -1  # FLCE_EINVAL: a shard needs the global lse


@pytest.mark.parametrize("dtype,N,V", [
    (torch.bfloat16, 1, 128256),   # one row, cluster of 4
    (torch.bfloat16, 1, 8),        # one 16-byte vector
    (torch.bfloat16, 3, 16),
    (torch.bfloat16, 2, 262144),   # the longest row a cluster of 8 holds (8 x 64 KiB)
    (torch.bfloat16, 2, 262152),   # one vector longer: streamed twice
    (torch.bfloat16, 3, 262143),   # rows inside blocks, one block too many: streamed twice
    (torch.float32, 2, 131072),    # the longest fp32 row a cluster holds
    (torch.bfloat16, 3, 1),        # one element per row
])
def test_no_lse_edge_shapes(lh, dtype, N, V):
    p = wl.random_ce(N, V, dtype, seed=N * 7 + V, ignore_frac=0.0)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    out = lh.ce_logits_fwd(logits, labels, -100, "sum")
    g = torch.tensor([0.5], device="cuda")
    grad = lh.ce_logits_bwd(logits, labels, None, out.n_valid, g, -100, "sum",
                            status=out.status)
    saved = lh.ce_logits_bwd(logits, labels, out.lse, out.n_valid, g, -100, "sum")
    torch.cuda.synchronize()
    lh.check_status(out.status)
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, "sum", grad_loss=0.5))
    _close_to_saved(grad, saved, dtype, 0.5)


@pytest.mark.parametrize("dtype,N,V", [(torch.bfloat16, 64, 50257), (torch.float32, 40, 4099),
                                       (torch.bfloat16, 70, 4096)])
@pytest.mark.parametrize("lse_saved", [False, True])
def test_grad_rows_at_other_offsets(lh, dtype, N, V, lse_saved):
    # the gradient buffer starts one element after a 16-byte boundary: its rows
    # sit at other offsets within their blocks than the logits rows, so the
    # register-streaming row kernel writes it
    p = wl.random_ce(N, V, dtype, seed=N + V, ignore_frac=0.1, reduction="mean")
    logits, labels = p.logits.cuda().contiguous(), p.labels.cuda()
    out = lh.ce_logits_fwd(logits, labels, -100, "mean")
    big = torch.full((N * V + 8,), float("nan"), dtype=dtype, device="cuda")
    gbuf = big[1:1 + N * V].view(N, V)
    g = torch.tensor([0.8], device="cuda")
    grad = lh.ce_logits_bwd(logits, labels, out.lse if lse_saved else None, out.n_valid, g,
                            -100, "mean", grad_logits=gbuf, status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert grad.data_ptr() == gbuf.data_ptr()
    assert torch.isnan(big[0]) and torch.all(torch.isnan(big[1 + N * V:]))  # nothing outside
    _check_grad(grad, oracle.ce_backward(p.logits, p.labels, -100, "mean", grad_loss=0.8))
