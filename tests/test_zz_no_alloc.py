"""The allocation-free CE forward (ce_logits_fwd_noalloc) against ce_logits_fwd.

ce_logits_fwd_noalloc serves callers that cannot call cudaMalloc (a runtime
that owns all device memory through its own pool, or a latency-critical loop
that must not risk the device-wide synchronisation of an allocation): its
per-row scratch is a static device array instead of a caller workspace.  This
file is collected last on purpose, so that a run stopping at the first failure
has already run every other test; it also passes when run alone.

Two calls in a row on different problems (the second smaller, so stale rows of
the first stay in the shared array) must each match the workspace entry point
and the fp64 oracle within the tolerances of the other CE tests: loss 1e-3
relative, per-row lse 5e-5 (1 + |lse|), n_valid exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(lh, abi, logits, labels, reduction):
    N, V = logits.shape
    dev = logits.device
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dt = abi.FLCE_BF16 if logits.dtype == torch.bfloat16 else abi.FLCE_F32
    red = abi.FLCE_SUM if reduction == "sum" else abi.FLCE_MEAN
    rc = abi.ce_logits_fwd_noalloc(logits.data_ptr(), dt, N, V, logits.stride(0),
                                   labels.data_ptr(), -100, red, -1, loss.data_ptr(),
                                   n_valid.data_ptr(), lse.data_ptr(), status.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    abi.check(rc, "ce_logits_fwd_noalloc")
    return loss, n_valid, lse, status


def test_noalloc_matches_workspace_entry_point():
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import _abi
    cases = [(wl.random_ce(5000, 20000, torch.bfloat16, seed=77), "mean"),
             (wl.random_ce(1200, 50257, torch.bfloat16, seed=78), "sum")]
    for p, red in cases:
        logits, labels = p.logits.cuda(), p.labels.cuda()
        ref = lh.ce_logits_fwd(logits, labels, -100, red)
        loss, n_valid, lse, status = _noalloc(lh, _abi, logits, labels, red)
        torch.cuda.synchronize()
        lh.check_status(status)
        lh.check_status(ref.status)
        assert int(n_valid.item()) == int(ref.n_valid.item())
        r = ref.loss.item()
        assert abs(loss.item() - r) <= 1e-3 * abs(r)
        a = lse.cpu().double().numpy()
        b = ref.lse.cpu().double().numpy()
        assert np.all(np.abs(a - b) <= 5e-5 * (1 + np.abs(b)))
        want = oracle.ce_forward(p.logits, p.labels, -100, red)
        assert int(n_valid.item()) == want["n_valid"]
        assert abs(loss.item() - want["loss"]) <= 1e-3 * abs(want["loss"])
        assert np.all(np.abs(a - want["lse"]) <= 5e-5 * (1 + np.abs(want["lse"])))


def test_noalloc_rejects_too_many_rows():
    from lm_head_linear_fwd_gb300 import _abi
    max_rows = 1 << 20
    logits = torch.empty((max_rows + 1, 8), dtype=torch.bfloat16, device="cuda")
    labels = torch.zeros(max_rows + 1, dtype=torch.int64, device="cuda")
    out = torch.empty(max_rows + 1, dtype=torch.float32, device="cuda")
    one = torch.empty(1, dtype=torch.float32, device="cuda")
    nv = torch.empty(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _abi.ce_logits_fwd_noalloc(logits.data_ptr(), 0, max_rows + 1, 8, 8, labels.data_ptr(),
                                    -100, 0, -1, one.data_ptr(), nv.data_ptr(), out.data_ptr(),
                                    st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -2  # FLCE_ESHAPE, nothing enqueued
