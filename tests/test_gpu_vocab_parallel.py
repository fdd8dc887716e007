"""Vocabulary-parallel FLCE on one GPU: three vocabulary shards run their
kernels one after the other; the cross-rank reductions (MAX / SUM of [N]
vectors, SUM of grad_H partials) are stood in for by torch reductions over the
shards.  Results must match the unsharded path and the fp64 oracle within the
tolerances of tests/test_gpu_flce.py."""
import numpy as np
import pytest
import torch

import oracle
import tolerances as tol
import workloads as wl

pytestmark = pytest.mark.gpu


def _grad_ok(got, want, name):
    mr = oracle.max_rel_err(got.float().cpu(), want)
    nw = oracle.normwise_err(got.float().cpu(), want)
    assert mr <= 2e-2 and nw <= 5e-3, (name, mr, nw)


@pytest.mark.parametrize("reduction,nlt,bias,dtype,chunk", [
    ("mean", None, True, torch.bfloat16, None),
    ("sum", 900, False, torch.bfloat16, None),
    ("sum", None, True, torch.float32, None),
    ("mean", None, True, torch.bfloat16, -512),   # each shard's backward in vocabulary slices
])
def test_three_vocab_shards_match_the_oracle(reduction, nlt, bias, dtype, chunk):
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import vocab_parallel as vp
    p = wl.random_flce(1000, 128, 3001, dtype, bias=bias, seed=21, reduction=reduction,
                       num_label_tokens=nlt, w_std=0.05)
    p.labels[:4] = torch.tensor([0, 1023, 1024, 3000])   # shard edges
    H, W, y = p.H.cuda(), p.W.cuda(), p.labels.cuda()
    b = p.bias.cuda() if bias else None
    V = p.V
    bounds = [(0, 1024), (1024, 2048), (2048, V)]
    ops = vp.CudaShardOps()
    st = lh.new_status("cuda")
    parts = [ops.partials(H, W[a:c], y, a, V, None if b is None else b[a:c], -100, st)
             for a, c in bounds]
    m_g = torch.stack([q[0] for q in parts]).amax(0)                     # all-reduce MAX
    s_g = torch.stack([ops.rescale(q[0], q[1], m_g) for q in parts]).sum(0)  # all-reduce SUM
    zy_g = torch.stack([q[2] for q in parts]).sum(0)                      # all-reduce SUM
    lse, loss, n_valid = ops.finish(m_g, s_g, zy_g, y, V, -100, reduction, nlt, st)
    g = torch.ones(1, device="cuda")
    grads = [ops.backward(H, W[a:c], y, a, V, None if b is None else b[a:c], -100, reduction, nlt,
                          lse, n_valid, g, chunk, True, True, st) for a, c in bounds]
    gH = torch.stack([q[0].float() for q in grads]).sum(0)                # all-reduce SUM
    gW = torch.cat([q[1] for q in grads])
    torch.cuda.synchronize()
    lh.check_status(st)
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt)
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt)
    assert int(n_valid.item()) == ref["n_valid"]
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    tol.check_flce_lse(lse, ref["lse"], p.H, p.W, p.bias)
    _grad_ok(gH, gr["grad_H"], "grad_H")
    _grad_ok(gW, gr["grad_W"], "grad_W")
    if bias:
        gb = torch.cat([q[2] for q in grads])
        _grad_ok(gb, gr["grad_b"], "grad_b")
    # and the unsharded library path gives the same lse
    full = lh.flce_fwd(H, W, y, b, -100, reduction, nlt)
    torch.cuda.synchronize()
    assert torch.allclose(full.lse, lse, rtol=0, atol=2e-4)


@pytest.mark.parametrize("bounds", [[(0, 1024), (1024, 2048), (2048, 3001)],
                                    [(0, 1001), (1001, 3001)]])
@pytest.mark.parametrize("inplace", [False, True])
def test_ce_on_logit_shards_matches_the_oracle(bounds, inplace):
    """Column shards of given logits (aligned and odd boundaries: both kernels)."""
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import vocab_parallel as vp
    c = wl.random_ce(600, 3001, torch.bfloat16, seed=77, reduction="mean")
    c.labels[:3] = torch.tensor([0, 1000, 3000])
    full = c.logits.cuda().contiguous()
    y = c.labels.cuda()
    V = c.V
    ops = vp.CudaLogitsShardOps()
    st = lh.new_status("cuda")
    parts = [ops.partials(full[:, a:b], None, y, a, V, None, -100, st) for a, b in bounds]
    m_g = torch.stack([q[0] for q in parts]).amax(0)
    s_g = torch.stack([ops.rescale(q[0], q[1], m_g) for q in parts]).sum(0)
    zy_g = torch.stack([q[2] for q in parts]).sum(0)
    lse, loss, n_valid = ops.finish(m_g, s_g, zy_g, y, V, -100, "mean", None, st)
    fwd = vp.ShardForward(loss, n_valid, lse, st)
    work = full.clone()
    grads = [vp.ce_backward(work[:, a:b], y, a, V, fwd, torch.tensor([0.5], device="cuda"),
                            reduction="mean", inplace_grad=inplace) for a, b in bounds]
    dz = torch.cat([g for g in grads], dim=1)
    torch.cuda.synchronize()
    lh.check_status(st)
    ref = oracle.ce_forward(c.logits, c.labels, -100, "mean")
    assert int(n_valid.item()) == ref["n_valid"]
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    got = lse.cpu().double().numpy()
    assert np.all(np.abs(got - ref["lse"]) <= 5e-5 * (1 + np.abs(ref["lse"])))
    _grad_ok(dz, oracle.ce_backward(c.logits, c.labels, -100, "mean", grad_loss=0.5), "dZ")
    if inplace:
        assert torch.equal(work, dz)


def test_empty_batch_on_shards():
    # a rank with no tokens: every shard step accepts N = 0; the loss is 0 and
    # the shards' weight and bias gradients are zero
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import vocab_parallel as vp
    V, D = 3001, 128
    W = torch.randn(V, D, device="cuda").to(torch.bfloat16)
    b = torch.randn(V, device="cuda").to(torch.bfloat16)
    H = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    bounds = [(0, 1024), (1024, V)]
    ops = vp.CudaShardOps()
    st = lh.new_status("cuda")
    parts = [ops.partials(H, W[a:c], y, a, V, b[a:c], -100, st) for a, c in bounds]
    m_g = torch.stack([q[0] for q in parts]).amax(0)
    s_g = torch.stack([ops.rescale(q[0], q[1], m_g) for q in parts]).sum(0)
    zy_g = torch.stack([q[2] for q in parts]).sum(0)
    lse, loss, n_valid = ops.finish(m_g, s_g, zy_g, y, V, -100, "mean", None, st)
    grads = [ops.backward(H, W[a:c], y, a, V, b[a:c], -100, "mean", None, lse, n_valid,
                          torch.ones(1, device="cuda"), None, True, True, st)
             for a, c in bounds]
    torch.cuda.synchronize()
    lh.check_status(st)
    assert loss.item() == 0.0 and n_valid.item() == 0 and lse.numel() == 0
    for gH, gW, gb in grads:
        assert gH.shape == (0, D)
        assert torch.count_nonzero(gW) == 0 and torch.count_nonzero(gb) == 0


class ThreadExchange:
    """All-reduce among the threads of one process, one thread per rank: each
    rank's max_ / sum_ deposits its tensor; once every rank has arrived, rank 0
    reduces the deposited tensors with torch (on the stream every rank
    launches on, so after all their kernels) and writes the result into each
    in place.  The host threads wait on each other; no kernel waits on another."""

    def __init__(self, n):
        import threading
        self.n = n
        self.barrier = threading.Barrier(n, timeout=120)
        self.slots = [None] * n
        self.local = threading.local()

    def _reduce(self, t, op):
        r = self.local.rank
        self.slots[r] = t
        self.barrier.wait()
        if r == 0:
            stack = torch.stack(self.slots)
            red = stack.amax(0) if op == "max" else stack.sum(0)
            for s in self.slots:
                s.copy_(red)
        self.barrier.wait()
        return t

    def max_(self, t):
        return self._reduce(t, "max")

    def sum_(self, t):
        return self._reduce(t, "sum")


def _run_ranks(n, fn):
    import threading
    ex = ThreadExchange(n)
    out, errs = [None] * n, []

    def body(r):
        try:
            ex.local.rank = r
            torch.cuda.set_device(0)
            out[r] = fn(r, ex)
        except BaseException as e:  # noqa: BLE001 - surfaced below
            errs.append(e)
            ex.barrier.abort()
    ts = [threading.Thread(target=body, args=(r,)) for r in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errs:
        raise errs[0]
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("reduction,nlt,bias", [("mean", None, True), ("sum", 700, False)])
def test_shipped_module_on_three_ranks_matches_the_oracle(reduction, nlt, bias):
    """vocab_parallel.forward / backward as shipped (their phases, collectives
    and dtypes: fp32 grad_H partials summed, then one rounding to bf16), three
    ranks as threads of this process with an in-process all-reduce."""
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import vocab_parallel as vp
    p = wl.random_flce(900, 256, 5003, torch.bfloat16, bias=bias, seed=23, reduction=reduction,
                       num_label_tokens=nlt, w_std=0.05)
    p.labels[:4] = torch.tensor([0, 1999, 2000, 5002])   # shard edges
    H, W, y = p.H.cuda(), p.W.cuda(), p.labels.cuda()
    b = p.bias.cuda() if bias else None
    V = p.V
    bounds = [(0, 2000), (2000, 3500), (3500, V)]
    g = torch.full((1,), 0.75, device="cuda")

    def rank(r, ex):
        a, c = bounds[r]
        bs = None if b is None else b[a:c]
        fwd = vp.forward(H, W[a:c], y, a, V, bs, reduction=reduction, num_label_tokens=nlt,
                         exchange=ex)
        gH, gW, gb = vp.backward(H, W[a:c], y, a, V, fwd, g, bs, reduction=reduction,
                                 num_label_tokens=nlt, exchange=ex)
        return fwd, gH, gW, gb
    res = _run_ranks(3, rank)
    for fwd, *_ in res:
        lh.check_status(fwd.status)
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt)
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt, grad_loss=0.75)
    for fwd, gH, _, _ in res:
        assert int(fwd.n_valid.item()) == ref["n_valid"]
        assert abs(fwd.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
        tol.check_flce_lse(fwd.lse, ref["lse"], p.H, p.W, p.bias)
        assert gH.dtype == torch.bfloat16
        _grad_ok(gH, gr["grad_H"], "grad_H")
    # every rank holds the same loss, lse and grad_H
    for fwd, gH, _, _ in res[1:]:
        assert torch.equal(fwd.lse, res[0][0].lse) and torch.equal(fwd.loss, res[0][0].loss)
        assert torch.equal(gH, res[0][1])
    _grad_ok(torch.cat([q[2] for q in res]), gr["grad_W"], "grad_W")
    if bias:
        _grad_ok(torch.cat([q[3] for q in res]), gr["grad_b"], "grad_b")
    # the fp32 sum rounded once is as close to the oracle as the unsharded
    # backward's grad_H (one bf16 rounding each)
    full = lh.flce_fwd(H, W, y, b, -100, reduction, nlt)
    fb = lh.flce_bwd(H, W, y, full.lse, full.n_valid, g, b, -100, reduction, nlt)
    torch.cuda.synchronize()
    nw_shard = oracle.normwise_err(res[0][1].float().cpu(), gr["grad_H"])
    nw_full = oracle.normwise_err(fb.grad_H.float().cpu(), gr["grad_H"])
    assert nw_shard <= 1.25 * nw_full + 2e-4, (nw_shard, nw_full)


@pytest.mark.parametrize("inplace", [False, True])
def test_shipped_ce_module_on_two_ranks_matches_the_oracle(inplace):
    """vocab_parallel.ce_forward / ce_backward as shipped, two ranks as threads."""
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import vocab_parallel as vp
    c = wl.random_ce(500, 4001, torch.bfloat16, seed=78, reduction="sum")
    c.labels[:2] = torch.tensor([1499, 1500])
    full = c.logits.cuda().contiguous()
    work = full.clone()
    y = c.labels.cuda()
    bounds = [(0, 1500), (1500, c.V)]

    def rank(r, ex):
        a, e = bounds[r]
        fwd = vp.ce_forward(work[:, a:e], y, a, c.V, reduction="sum", exchange=ex)
        dz = vp.ce_backward(work[:, a:e], y, a, c.V, fwd, torch.ones(1, device="cuda"),
                            reduction="sum", inplace_grad=inplace)
        return fwd, dz
    res = _run_ranks(2, rank)
    ref = oracle.ce_forward(c.logits, c.labels, -100, "sum")
    for fwd, _ in res:
        lh.check_status(fwd.status)
        assert int(fwd.n_valid.item()) == ref["n_valid"]
        assert abs(fwd.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
        assert np.all(np.abs(fwd.lse.cpu().double().numpy() - ref["lse"]) <=
                      tol.CE_LSE * (1 + np.abs(ref["lse"])))
    dz = torch.cat([q[1] for q in res], dim=1)
    _grad_ok(dz, oracle.ce_backward(c.logits, c.labels, -100, "sum"), "dZ")
    if inplace:
        assert torch.equal(work, dz)
