"""Peak extra device memory of each path against the bound the hot-path
specification sets: at most one [chunk, V] fp32 tile plus the outputs, with
the chunk fixed at 2048 rows (Automodel PR #2996, first commit message and
"Motivation": the fp32 transient of its chunked loss is chunk_size x V x 4
bytes), whatever chunk the library picks for itself
(torch.cuda.max_memory_allocated over the calls, minus what was allocated
before them; every buffer the library uses comes from the caller, so the
Python API's allocations are all there is)."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lh():
    import lm_head_linear_fwd_gb300 as m
    return m


def _peak_extra(fn):
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    keep = fn()
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    del keep
    return extra


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("N,D,V,bias", [(4096, 1024, 50304, True), (8192, 4096, 128256, False)],
                         ids=["4096x1024x50304", "llama3_8b"])
def test_flce_peak_extra_memory(lh, fused, N, D, V, bias):
    p = wl.random_flce(N, D, V, torch.bfloat16, bias=bias, seed=71, device="cuda")
    H, W, b, y = p.H, p.W, p.bias, p.labels

    def run():
        if fused:
            return lh.flce_fwd_bwd(H, W, y, b, -100, "mean")
        out = lh.flce_fwd(H, W, y, b, -100, "mean")
        return out, lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b,
                                -100, "mean")
    extra = _peak_extra(run)
    # grad_H, grad_W, grad_b, lse, per-row losses, scalars
    outputs = N * D * 2 + V * D * 4 + (V * 4 if bias else 0) + N * 4 * 2 + 64
    bound = 2048 * V * 4 + outputs
    assert extra <= bound, (extra, bound)


def test_ce_in_place_peak_extra_memory(lh):
    c = wl.random_ce(4096, 32768, torch.bfloat16, seed=72, device="cuda")
    logits, y = c.logits.contiguous(), c.labels

    def run():
        out = lh.ce_logits_fwd(logits, y, -100, "sum")
        lh.ce_logits_bwd(logits, y, out.lse, out.n_valid, torch.ones(1, device="cuda"),
                         inplace_grad=True)
        return out
    extra = _peak_extra(run)
    # the lse and the per-row scratch (4 bytes per row each) plus a few scalars
    assert extra <= 2 * 4096 * 4 + (1 << 16), extra
