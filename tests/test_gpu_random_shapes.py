"""Seeded random shapes for both paths (recomputing and fused FLCE, CE on
logits) against the fp64 oracle: sizes drawn across tile, chunk and vector
boundaries, random dtype, bias, reduction and chunk.  Tolerances as in
tests/test_gpu_flce.py and tests/test_gpu_ce_logits.py (tests/tolerances.py):
the per-row lse of both FLCE paths is held to 2e-5 (1 + |lse|) for bf16, so a
lost 256-column vocabulary tile fails, also at the large vocabularies of the
third draw."""
import numpy as np
import pytest
import torch

import oracle
import tolerances as tol
import workloads as wl

pytestmark = pytest.mark.gpu

CASES = []
_rng = np.random.default_rng(2026)
for i in range(12):
    CASES.append(dict(
        N=int(_rng.integers(1, 1500)),
        D=int(_rng.integers(1, 80)) * 8,
        V=int(_rng.integers(2, 9000)),
        dtype=torch.bfloat16 if _rng.random() < 0.75 else torch.float32,
        bias=bool(_rng.random() < 0.5),
        reduction=str(_rng.choice(["sum", "mean"])),
        nlt=None if _rng.random() < 0.7 else int(_rng.integers(0, 2000)),
        chunk=None if _rng.random() < 0.5 else int(_rng.integers(1, 8)) * 128,
        seed=1000 + i))


# a second draw: larger vocabularies, ignored fractions up to one half, and
# row counts around multiples of the 128-row tile
_rng2 = np.random.default_rng(7)
for i in range(8):
    CASES.append(dict(
        N=int(_rng2.integers(1, 12)) * 128 + int(_rng2.integers(-2, 3)) + 2,
        D=int(_rng2.integers(1, 40)) * 16,
        V=int(_rng2.integers(9000, 40000)),
        dtype=torch.bfloat16,
        bias=bool(_rng2.random() < 0.5),
        reduction=str(_rng2.choice(["sum", "mean"])),
        nlt=None,
        chunk=None if _rng2.random() < 0.5 else int(_rng2.integers(1, 6)) * 128,
        ignore=float(_rng2.choice([0.0, 0.1, 0.5])),
        seed=2000 + i))


# a third draw: vocabularies of 1.2e5 to 1.6e5 words (470 to 625 tiles of 256
# columns, the range of the Llama3-8B and long packed heads), few rows
_rng3 = np.random.default_rng(128256)
for i in range(4):
    CASES.append(dict(
        N=int(_rng3.integers(1, 400)),
        D=int(_rng3.integers(1, 24)) * 8,
        V=int(_rng3.integers(120000, 160000)),
        dtype=torch.bfloat16 if i < 3 else torch.float32,
        bias=bool(i % 2),
        reduction=str(_rng3.choice(["sum", "mean"])),
        nlt=None,
        chunk=None if i % 2 else 128,
        seed=3000 + i))


def _grad_ok(got, want, name):
    mr = oracle.max_rel_err(got.float().cpu(), want)
    nw = oracle.normwise_err(got.float().cpu(), want)
    assert mr <= 2e-2 and nw <= 5e-3, (name, mr, nw)


@pytest.mark.parametrize("case", CASES, ids=[f"{c['N']}x{c['D']}x{c['V']}" for c in CASES])
def test_flce_random_shape(case):
    import lm_head_linear_fwd_gb300 as lh
    p = wl.random_flce(case["N"], case["D"], case["V"], case["dtype"], bias=case["bias"],
                       seed=case["seed"], ignore_frac=case.get("ignore", 0.1),
                       reduction=case["reduction"], num_label_tokens=case["nlt"], w_std=0.05)
    H, W, y = p.H.cuda(), p.W.cuda(), p.labels.cuda()
    b = p.bias.cuda() if p.bias is not None else None
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens)
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, p.reduction, p.num_label_tokens)
    out = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens)
    bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b, -100,
                     p.reduction, p.num_label_tokens, case["chunk"])
    fo, fb = lh.flce_fwd_bwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, case["chunk"])
    torch.cuda.synchronize()
    lh.check_status(out.status)
    lh.check_status(fo.status)
    for o in (out, fo):
        assert int(o.n_valid.item()) == ref["n_valid"]
        assert abs(o.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"]) + 1e-6
    tol.check_flce_lse(out.lse, ref["lse"], p.H, p.W, p.bias, what="lse (flce_fwd)")
    tol.check_flce_lse(fo.lse, ref["lse"], p.H, p.W, p.bias, what="lse (flce_fwd_bwd)")
    if ref["loss"] == 0.0:
        return
    for g in (bw, fb):
        _grad_ok(g.grad_H, gr["grad_H"], "grad_H")
        _grad_ok(g.grad_W, gr["grad_W"], "grad_W")
        if b is not None:
            _grad_ok(g.grad_bias, gr["grad_b"], "grad_b")


@pytest.mark.parametrize("case", CASES[:8], ids=[f"{c['N']}x{c['V']}" for c in CASES[:8]])
def test_ce_random_shape(case):
    import lm_head_linear_fwd_gb300 as lh
    # a row stride a few elements over V, and for some cases a first column
    # inside a 16-byte block (a column slice of a wider buffer)
    c0 = int(case["seed"] % 5)
    ld = case["V"] + c0 + (0 if case["seed"] % 2 else int(case["seed"] % 13))
    c = wl.random_ce(case["N"], ld, case["dtype"], seed=case["seed"],
                     reduction=case["reduction"], num_label_tokens=case["nlt"])
    c.logits = c.logits[:, c0:c0 + case["V"]]
    c.labels = torch.where(c.labels >= case["V"], c.labels % case["V"], c.labels)
    logits, y = c.logits.cuda(), c.labels.cuda()
    out = lh.ce_logits_fwd(logits, y, -100, c.reduction, c.num_label_tokens)
    grad = lh.ce_logits_bwd(logits, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), -100,
                            c.reduction, c.num_label_tokens)
    torch.cuda.synchronize()
    ref = oracle.ce_forward(c.logits, c.labels, -100, c.reduction, c.num_label_tokens)
    assert int(out.n_valid.item()) == ref["n_valid"]
    assert abs(out.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"]) + 1e-6
    lse = out.lse.cpu().double().numpy()
    assert np.all(np.abs(lse - ref["lse"]) <= 5e-5 * (1 + np.abs(ref["lse"])))
    # the same gradient without the saved lse (formed again in the backward)
    grad2 = lh.ce_logits_bwd(logits, y, None, out.n_valid, torch.ones(1, device="cuda"), -100,
                             c.reduction, c.num_label_tokens, status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    # and forward and backward in one call
    o3, grad3 = lh.ce_logits_fwd_bwd(logits, y, -100, c.reduction, c.num_label_tokens,
                                     status=out.status)
    torch.cuda.synchronize()
    lh.check_status(out.status)
    assert int(o3.n_valid.item()) == ref["n_valid"]
    assert abs(o3.loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"]) + 1e-6
    if ref["loss"] != 0.0:
        want = oracle.ce_backward(c.logits, c.labels, -100, c.reduction, c.num_label_tokens)
        _grad_ok(grad, want, "dZ")
        _grad_ok(grad2, want, "dZ without a saved lse")
        _grad_ok(grad3, want, "dZ in one call")
