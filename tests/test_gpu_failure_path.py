"""The failure path of the bounded waits, without a GPU fault: a wait that
nothing satisfies gives up after a short limit, FLCE_ETIMEOUT reaches the
status word, and the context keeps working (the next library call succeeds)."""
import time

import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import _abi
    st = lh.new_status("cuda")
    t0 = time.perf_counter()
    rc = _abi.flce_wait_selftest(st.data_ptr(), 20_000_000, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == -9          # FLCE_ETIMEOUT
    assert 0.01 <= elapsed < 2.0
    with pytest.raises(lh.FlceError):
        lh.check_status(st)
    # the context is intact: an ordinary call still runs and is correct
    p = wl.random_ce(64, 1000, torch.bfloat16, seed=1)
    out = lh.ce_logits_fwd(p.logits.cuda(), p.labels.cuda())
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert torch.isfinite(out.loss).all()
