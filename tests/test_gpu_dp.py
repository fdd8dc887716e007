"""Data-parallel sharding with the CUDA kernels on one GPU: shards run one
after the other with the global valid count as num_label_tokens; their losses
and gradients must add up to the single-call mean."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def test_count_valid_kernel():
    from lm_head_linear_fwd_gb300 import dp
    y = wl.uniform_labels(10000, 5000, seed=3, device="cuda")
    y[::7] = -100
    y[5] = 5000   # out of range: not counted
    y[6] = -3
    want = int(((y != -100) & (y >= 0) & (y < 5000)).sum())
    assert int(dp.local_valid_count(y, 5000).item()) == want


def test_shards_add_up_to_the_global_mean():
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import dp
    p = wl.random_flce(1000, 256, 3001, torch.bfloat16, seed=17, reduction="mean")
    H, W, y = p.H.cuda(), p.W.cuda(), p.labels.cuda()
    total = dp.global_num_label_tokens(y, p.V)   # no process group: the local count
    one = torch.ones(1, device="cuda")
    full_o = lh.flce_fwd(H, W, y, None, -100, "mean")
    full_b = lh.flce_bwd(H, W, y, full_o.lse, full_o.n_valid, one, None, -100, "mean")
    loss, gW = 0.0, torch.zeros_like(full_b.grad_W)
    for rank in range(3):
        a, b = dp.shard_rows(p.N, rank, 3)
        o = lh.flce_fwd(H[a:b], W, y[a:b], None, -100, "sum", total)
        lh.flce_bwd(H[a:b], W, y[a:b], o.lse, o.n_valid, one, None, -100, "sum", total,
                    grad_W=gW, accumulate_grad_W=True, want_grad_H=False)
        loss += o.loss.item()
    torch.cuda.synchronize()
    assert abs(loss - full_o.loss.item()) <= 1e-5 * abs(full_o.loss.item())
    assert oracle.normwise_err(gW.cpu(), full_b.grad_W.cpu().double().numpy()) <= 1e-5


def test_mask_packed_labels_matches_the_oracle():
    """The kernel against the oracle's packed-document masking (padding and the
    last token of each document ignored), bit-exact, on rows laid out like the
    long packed workload (a padding tail, four documents at random cuts) and
    on rows with padding first, one-token documents and no padding."""
    import lm_head_linear_fwd_gb300 as lh
    B, T, V = 4, 4096, 151936
    doc = torch.zeros(B, T, dtype=torch.int64)
    rng = torch.Generator().manual_seed(7)
    pad = 327
    labels = torch.randint(0, V, (B, T), generator=rng)
    for r in range(B):
        cuts = sorted((torch.randperm(T - pad - 2, generator=rng)[:3] + 1).tolist())
        start = 0
        for k, e in enumerate(cuts + [T - pad]):
            doc[r, start:e] = k + 1
            start = e
    doc2 = torch.tensor([[0, 0, 1, 2, 2, 3, 4, 4], [5, 5, 5, 5, 5, 5, 5, 5]], dtype=torch.int64)
    labels2 = torch.randint(0, V, (2, 8), generator=rng)
    for d, y in ((doc, labels), (doc2, labels2)):
        out = lh.mask_packed_labels(y.cuda(), d.cuda())
        torch.cuda.synchronize()
        want = oracle.packed_document_labels(y, d)
        assert np.array_equal(out.cpu().numpy(), want)
