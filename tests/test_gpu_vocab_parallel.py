"""Vocabulary-parallel FLCE on one GPU: three vocabulary shards run their
kernels one after the other; the cross-rank reductions (MAX / SUM of [N]
vectors, SUM of grad_H partials) are stood in for by torch reductions over the
shards.  Results must match the unsharded path and the fp64 oracle within the
tolerances of tests/test_gpu_flce.py."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def _grad_ok(got, want, name):
    mr = oracle.max_rel_err(got.float().cpu(), want)
    nw = oracle.normwise_err(got.float().cpu(), want)
    assert mr <= 2e-2 and nw <= 5e-3, (name, mr, nw)


@pytest.mark.parametrize("reduction,nlt,bias,dtype", [("mean", None, True, torch.bfloat16),
                                                      ("sum", 900, False, torch.bfloat16),
                                                      ("sum", None, True, torch.float32)])
def test_three_vocab_shards_match_the_oracle(reduction, nlt, bias, dtype):
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
                          lse, n_valid, g, None, True, True, st) for a, c in bounds]
    gH = torch.stack([q[0].float() for q in grads]).sum(0)                # all-reduce SUM
    gW = torch.cat([q[1] for q in grads])
    torch.cuda.synchronize()
    lh.check_status(st)
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt)
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, reduction, nlt)
    assert int(n_valid.item()) == ref["n_valid"]
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    got_lse = lse.cpu().double().numpy()
    assert np.max(np.abs(got_lse - ref["lse"]) / (1 + np.abs(ref["lse"]))) <= 2e-3
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
