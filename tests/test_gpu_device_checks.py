"""The debug build with device-side index checks (FLCE_DEVICE_CHECKS=1).

The test compiles it (``build.build(checked=True)`` writes libflce_checked.so
beside libflce.so), opens it beside the ordinary build, and runs the package's
Python API against each library in turn by swapping the handle the API calls
through.  Every path must leave the status word at 0 (no index left its
range) and give results bit-identical to the ordinary build: the checks add no
arithmetic.  flce_bounds_selftest shows that a failed check is recorded in the
checked build (FLCE_EBOUNDS) and compiled out of the ordinary one.  The debug
build stands in for a memory checker, which this GPU pool does not offer.
"""
import contextlib

import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    from lm_head_linear_fwd_gb300 import _abi, build
    checked = _abi.open_library(build.build(checked=True))
    return _abi.load(), checked


@contextlib.contextmanager
def _using(lib):
    from lm_head_linear_fwd_gb300 import _abi
    old = _abi._lib
    _abi._lib = lib
    try:
        yield
    finally:
        _abi._lib = old


def test_build_flags_and_bounds_selftest(libs):
    ordinary, checked = libs
    assert ordinary.flce_device_checks() == 0
    assert checked.flce_device_checks() == 1
    for lib, want in ((ordinary, 0), (checked, -10)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert lib.flce_bounds_selftest(st.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == want


def _ce_cases():
    # (dtype, N, V, ld): the bulk-copy ring, rows that start and end inside
    # 16-byte blocks, and for the no-lse backward and the one-call forward and
    # backward clusters of 1, 2 and 4 and the twice-streamed rows
    return [(torch.bfloat16, 300, 5000, 5000), (torch.bfloat16, 77, 1003, 1011),
            (torch.float32, 64, 4100, 4104), (torch.bfloat16, 64, 128256, 128256),
            (torch.bfloat16, 4, 300000, 300000), (torch.bfloat16, 40, 50257, 50257),
            (torch.bfloat16, 3, 262143, 262143)]


def _run_ce(lh, dtype, N, V, ld):
    p = wl.random_ce(N, V, dtype, seed=N + V, reduction="mean", ld=ld)
    logits, labels = p.logits.cuda(), p.labels.cuda()
    st = lh.new_status("cuda")
    o = lh.ce_logits_fwd(logits, labels, -100, "mean", want_rows=True, status=st)
    g = torch.tensor([0.9], device="cuda")
    saved = lh.ce_logits_bwd(logits, labels, o.lse, o.n_valid, g, -100, "mean", status=st)
    nolse = lh.ce_logits_bwd(logits, labels, None, o.n_valid, g, -100, "mean", status=st)
    fo, fg = lh.ce_logits_fwd_bwd(logits, labels, -100, "mean", None, g, want_lse=True,
                                  status=st)
    torch.cuda.synchronize()
    return st, [o.loss, o.lse, o.loss_rows, o.n_valid, saved, nolse, fo.loss,
                fo.lse.nan_to_num(0.0), fg]


def _run_flce(lh, dtype, N, D, V, bias):
    p = wl.random_flce(N, D, V, dtype, bias=bias, seed=N + D + V, reduction="mean")
    H, W, y = p.H.cuda(), p.W.cuda(), p.labels.cuda()
    b = p.bias.cuda() if bias else None
    st = lh.new_status("cuda")
    o = lh.flce_fwd(H, W, y, b, -100, "mean", status=st)
    g = torch.tensor([1.1], device="cuda")
    r = lh.flce_bwd(H, W, y, o.lse, o.n_valid, g, b, -100, "mean", None, 128, status=st)
    fo, fr = lh.flce_fwd_bwd(H, W, y, b, -100, "mean", status=st)
    torch.cuda.synchronize()
    outs = [o.loss, o.lse, r.grad_H, r.grad_W, fo.loss, fr.grad_H, fr.grad_W]
    if bias:
        outs += [r.grad_bias, fr.grad_bias]
    return st, outs


def _same_under_both(libs, fn, *args):
    import lm_head_linear_fwd_gb300 as lh
    ordinary, checked = libs
    results = []
    for lib in (ordinary, checked):
        with _using(lib):
            st, outs = fn(lh, *args)
            assert int(st.item()) == 0, lh.FlceError(int(st.item()), "device status")
            results.append([t.clone() for t in outs])
    for a, b in zip(*results):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,N,V,ld", _ce_cases())
def test_ce_paths_pass_every_check(libs, dtype, N, V, ld):
    _same_under_both(libs, _run_ce, dtype, N, V, ld)


@pytest.mark.parametrize("dtype,N,D,V,bias", [
    (torch.bfloat16, 700, 256, 5000, True),   # tile edges in M, N; grad_W on CTA pairs
    (torch.float32, 256, 128, 1000, False),   # tf32 path with its transposes
    (torch.bfloat16, 96, 768, 32777, False),  # split-K grad_H, odd vocabulary
])
def test_flce_paths_pass_every_check(libs, dtype, N, D, V, bias):
    _same_under_both(libs, _run_flce, dtype, N, D, V, bias)
