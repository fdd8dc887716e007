"""Pins of the fp64 CPU oracle against things other than itself.

Each pin is independent of the oracle's own code: hand-derived closed forms
(tests/golden/closed_forms.json), a loop-only restatement without the
max-subtraction, PyTorch's float64 ``F.cross_entropy`` and its autograd (the
routine the Automodel PR #2996 "Proof" section checks its chunked path
against), central finite differences, and invariants of softmax
cross-entropy.  The last tests plant mistakes in the oracle and check that the
pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bruteforce
from oracle import lm_head_ce as olc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _rand(N, D, V, seed, bias=True, ignore=(1,)):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.7
    b = rng.standard_normal(V) * 0.3 if bias else None
    y = rng.integers(0, V, N)
    for i in ignore:
        if i < N:
            y[i] = -100
    return H, W, b, y


# ------------------------------------------------------------------ golden closed forms

def test_golden_probs_1234():
    g = json.load(open(GOLDEN))["ce_probs_1234"]
    Z = np.log(np.array(g["logits_as_log_of"], dtype=np.float64))
    y = np.array(g["labels"])
    f = oracle.ce_forward(Z, y, -100, "sum")
    assert f["n_valid"] == g["n_valid"]
    np.testing.assert_allclose(f["lse"], g["lse"], rtol=1e-14)
    np.testing.assert_allclose(f["loss_rows"], g["loss_rows"], rtol=1e-14, atol=1e-15)
    assert f["loss"] == pytest.approx(g["loss_sum"], rel=1e-14)
    fm = oracle.ce_forward(Z, y, -100, "mean")
    assert fm["loss"] == pytest.approx(g["loss_mean"], rel=1e-14)
    dZ = oracle.ce_backward(Z, y, -100, "sum")
    np.testing.assert_allclose(dZ, g["dZ_sum"], atol=1e-14)
    dZm = oracle.ce_backward(Z, y, -100, "mean", grad_loss=2.0)  # mean halves, g=2 doubles
    np.testing.assert_allclose(dZm, g["dZ_sum"], atol=1e-14)


def test_golden_peaked_row():
    g = json.load(open(GOLDEN))["ce_peaked_row"]
    Z = np.array([[g["L"], 0.0, 0.0]])
    f = oracle.ce_forward(Z, np.array([0]), -100, "sum")
    assert f["loss"] == pytest.approx(g["loss"], rel=1e-13)


def test_golden_zero_weight_flce():
    g = json.load(open(GOLDEN))["flce_zero_weight"]
    H = np.array(g["H"])
    V = g["V"]
    W = np.zeros((V, H.shape[1]))
    b = np.zeros(V)
    y = np.array(g["labels"])
    f = oracle.flce_forward(H, W, b, y, -100, "sum")
    assert f["n_valid"] == g["n_valid"]
    assert f["loss"] == pytest.approx(g["loss_sum"], rel=1e-14)
    gr = oracle.flce_backward(H, W, b, y, -100, "sum")
    np.testing.assert_allclose(gr["grad_b"], g["grad_b"], atol=1e-14)
    np.testing.assert_allclose(gr["grad_W"], g["grad_W"], atol=1e-14)
    np.testing.assert_array_equal(gr["grad_H"], 0.0)


# --------------------------------------------------------------- closed forms at size

@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_zero_weight_closed_form(reduction):
    N, D, V = 40, 6, 1000
    H, _, _, y = _rand(N, D, V, 3, ignore=(0, 5, 7))
    W = np.zeros((V, D))
    f = oracle.flce_forward(H, W, None, y, -100, reduction)
    nv = N - 3
    assert f["n_valid"] == nv
    want = nv * math.log(V) if reduction == "sum" else math.log(V)
    assert f["loss"] == pytest.approx(want, rel=1e-13)
    g = 0.75
    dZ = oracle.ce_backward(np.zeros((N, V)), y, -100, reduction, grad_loss=g)
    sc = g * (1.0 if reduction == "sum" else 1.0 / nv)
    want_dZ = np.full((N, V), 1.0 / V) * sc
    for i in range(N):
        if y[i] == -100:
            want_dZ[i] = 0
        else:
            want_dZ[i, y[i]] -= sc
    np.testing.assert_allclose(dZ, want_dZ, atol=1e-15)


def test_constant_rows_give_ln_V():
    V = 777
    Z = np.full((5, V), 3.25)
    y = np.array([0, 1, 776, 400, -100])
    f = oracle.ce_forward(Z, y, -100, "sum")
    np.testing.assert_allclose(f["loss_rows"][:4], math.log(V), rtol=1e-13)
    assert f["loss_rows"][4] == 0.0


def test_large_logits_do_not_overflow():
    Z = np.array([[1000.0, 999.0, -1000.0], [-5000.0, -5001.0, -5002.0]])
    f = oracle.ce_forward(Z, np.array([0, 2]), -100, "sum")
    np.testing.assert_allclose(f["loss_rows"][0], math.log1p(math.exp(-1.0) + math.exp(-2000.0)),
                               rtol=1e-13)
    np.testing.assert_allclose(f["loss_rows"][1], 2.0 + math.log(1 + math.exp(-1) + math.exp(-2)),
                               rtol=1e-11)  # |Z| ~ 5000: ~5000 ulp of cancellation


# ------------------------------------------------------------ loop-only restatement

@pytest.mark.parametrize("reduction,nlt", [("sum", None), ("mean", None), ("sum", 7)])
def test_bruteforce_flce(reduction, nlt):
    N, D, V = 6, 5, 13
    H, W, b, y = _rand(N, D, V, 11, ignore=(2,))
    loss, nv, gH, gW, gb = bruteforce.flce(H.tolist(), W.tolist(), b.tolist(), y.tolist(),
                                           -100, reduction, nlt, grad_loss=1.3)
    f = oracle.flce_forward(H, W, b, y, -100, reduction, nlt)
    gr = oracle.flce_backward(H, W, b, y, -100, reduction, nlt, grad_loss=1.3)
    assert f["n_valid"] == nv
    assert f["loss"] == pytest.approx(loss, rel=1e-13)
    np.testing.assert_allclose(gr["grad_H"], gH, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gr["grad_W"], gW, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gr["grad_b"], gb, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------- PyTorch float64 library routine

@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_matches_torch_cross_entropy(reduction):
    N, V = 64, 301
    rng = np.random.default_rng(5)
    Z = rng.standard_normal((N, V)) * 3
    y = rng.integers(0, V, N)
    y[::7] = -100
    Zt = torch.tensor(Z, requires_grad=True)
    ref = F.cross_entropy(Zt, torch.tensor(y), ignore_index=-100, reduction=reduction)
    ref.backward(torch.tensor(0.5, dtype=torch.float64))
    f = oracle.ce_forward(Z, y, -100, reduction)
    assert f["loss"] == pytest.approx(ref.item(), rel=1e-13)
    dZ = oracle.ce_backward(Z, y, -100, reduction, grad_loss=0.5)
    np.testing.assert_allclose(dZ, Zt.grad.numpy(), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("bias", [False, True])
def test_flce_matches_torch_autograd(bias):
    N, D, V = 37, 24, 211
    H, W, b, y = _rand(N, D, V, 9, bias=bias, ignore=(0, 3, 30))
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True) if bias else None
    Z = Ht @ Wt.T + (bt if bias else 0)
    nlt = 50
    ref = F.cross_entropy(Z, torch.tensor(y), ignore_index=-100, reduction="sum") / nlt
    ref.backward()
    f = oracle.flce_forward(H, W, b, y, -100, "sum", nlt)
    gr = oracle.flce_backward(H, W, b, y, -100, "sum", nlt)
    assert f["loss"] == pytest.approx(ref.item(), rel=1e-13)
    np.testing.assert_allclose(gr["grad_H"], Ht.grad.numpy(), rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(gr["grad_W"], Wt.grad.numpy(), rtol=1e-11, atol=1e-15)
    if bias:
        np.testing.assert_allclose(gr["grad_b"], bt.grad.numpy(), rtol=1e-11, atol=1e-15)


# ------------------------------------------------------------- finite differences

def _fd(fun, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = fun()
        x[i] = old - eps
        fm = fun()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


def test_finite_differences_flce():
    N, D, V = 5, 4, 7
    H, W, b, y = _rand(N, D, V, 21, ignore=(1,))
    loss = lambda: oracle.flce_forward(H, W, b, y, -100, "mean")["loss"]  # noqa: E731
    gr = oracle.flce_backward(H, W, b, y, -100, "mean")
    np.testing.assert_allclose(gr["grad_H"], _fd(loss, H), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(gr["grad_W"], _fd(loss, W), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(gr["grad_b"], _fd(loss, b), rtol=1e-6, atol=1e-9)


def test_finite_differences_ce():
    rng = np.random.default_rng(4)
    Z = rng.standard_normal((4, 9))
    y = np.array([3, -100, 8, 0])
    loss = lambda: oracle.ce_forward(Z, y, -100, "sum", num_label_tokens=3)["loss"]  # noqa: E731
    dZ = oracle.ce_backward(Z, y, -100, "sum", num_label_tokens=3)
    np.testing.assert_allclose(dZ, _fd(loss, Z), rtol=1e-6, atol=1e-9)


# --------------------------------------------------------------------- invariants

def test_invariants():
    N, D, V = 30, 8, 97
    H, W, b, y = _rand(N, D, V, 17, ignore=(2, 9))
    f = oracle.flce_forward(H, W, b, y, -100, "sum")
    assert np.all(f["loss_rows"] >= 0)
    dZ = oracle.ce_backward(oracle.flce_logits(H, W, b, np.arange(N)), y, -100, "sum")
    np.testing.assert_allclose(dZ.sum(axis=1), 0.0, atol=1e-14)
    assert np.all(dZ[[2, 9]] == 0)
    gr = oracle.flce_backward(H, W, b, y, -100, "sum")
    np.testing.assert_allclose(gr["grad_b"].sum(), 0.0, atol=1e-13)
    np.testing.assert_allclose(gr["grad_W"].sum(axis=0), 0.0, atol=1e-12)
    assert np.all(gr["grad_H"][[2, 9]] == 0)


def test_shift_invariance():
    N, D, V = 12, 5, 31
    H, W, b, y = _rand(N, D, V, 23)
    f0 = oracle.flce_forward(H, W, b, y, -100, "sum")
    f1 = oracle.flce_forward(H, W, b + 17.5, y, -100, "sum")
    assert f1["loss"] == pytest.approx(f0["loss"], rel=1e-12)
    g0 = oracle.flce_backward(H, W, b, y, -100, "sum")
    g1 = oracle.flce_backward(H, W, b + 17.5, y, -100, "sum")
    np.testing.assert_allclose(g1["grad_H"], g0["grad_H"], atol=1e-12)
    Z = np.random.default_rng(1).standard_normal((N, V))
    shift = np.arange(N)[:, None] * 3.0
    np.testing.assert_allclose(oracle.ce_backward(Z + shift, y, -100, "sum"),
                               oracle.ce_backward(Z, y, -100, "sum"), atol=1e-13)


def test_grad_W_is_linear_in_row_blocks():
    N, D, V = 40, 6, 53
    H, W, b, y = _rand(N, D, V, 31, ignore=(4, 33))
    full = oracle.flce_backward(H, W, b, y, -100, "mean")
    nv = int((y != -100).sum())
    acc = np.zeros((V, D))
    for r0 in range(0, N, 13):
        rows = np.arange(r0, min(N, r0 + 13))
        part = oracle.flce_backward(H, W, b, y, -100, "mean", rows=rows, n_valid_total=nv,
                                    grad_W_init=acc)
        acc = part["grad_W"]
        np.testing.assert_allclose(part["grad_H"], full["grad_H"][rows], atol=1e-14)
    np.testing.assert_allclose(acc, full["grad_W"], atol=1e-13)


# ------------------------------------------------------------------- zero guards

@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_all_ignored_gives_zero(reduction):
    N, D, V = 8, 4, 11
    H, W, b, _ = _rand(N, D, V, 2)
    y = np.full(N, -100)
    f = oracle.flce_forward(H, W, b, y, -100, reduction)
    assert f["loss"] == 0.0 and f["n_valid"] == 0
    gr = oracle.flce_backward(H, W, b, y, -100, reduction)
    for k in ("grad_H", "grad_W", "grad_b"):
        assert np.all(gr[k] == 0)


def test_zero_num_label_tokens_guard():
    N, D, V = 8, 4, 11
    H, W, b, y = _rand(N, D, V, 2)
    f = oracle.flce_forward(H, W, b, y, -100, "sum", num_label_tokens=0)
    assert f["loss"] == 0.0 and f["n_valid"] == N - 1
    gr = oracle.flce_backward(H, W, b, y, -100, "sum", num_label_tokens=0)
    for k in ("grad_H", "grad_W", "grad_b"):
        assert np.all(gr[k] == 0)


def test_num_label_tokens_overrides_divisor():
    N, D, V = 10, 3, 9
    H, W, b, y = _rand(N, D, V, 8)
    s = oracle.flce_forward(H, W, b, y, -100, "sum")["loss"]
    for red in ("sum", "mean"):
        assert oracle.flce_forward(H, W, b, y, -100, red, 4)["loss"] == pytest.approx(s / 4, rel=1e-14)


def test_ignore_index_inside_vocab_is_ignored():
    Z = np.random.default_rng(0).standard_normal((3, 5))
    f = oracle.ce_forward(Z, np.array([2, 4, 0]), ignore_index=4)
    assert f["n_valid"] == 2 and f["loss_rows"][1] == 0.0


def test_out_of_range_label_raises():
    with pytest.raises(ValueError):
        oracle.ce_forward(np.zeros((2, 5)), np.array([1, 5]))
    with pytest.raises(ValueError):
        oracle.ce_forward(np.zeros((2, 5)), np.array([-1, 0]))


def test_bf16_inputs_are_widened_exactly():
    t = torch.tensor([[1.0, 2.0, 3.0]], dtype=torch.float32).to(torch.bfloat16) * 1.01
    Z = olc._f64(t)
    assert Z.dtype == np.float64
    assert np.all(Z == t.float().numpy().astype(np.float64))


# ------------------------------------------------------- planted mistakes are caught

def _golden_probs_ok():
    try:
        test_golden_probs_1234()
        return True
    except AssertionError:
        return False


def test_planted_lse_without_max_is_caught(monkeypatch):
    monkeypatch.setattr(olc, "logsumexp_rows",
                        lambda Z: np.log(np.exp(Z - Z.max(axis=1)[:, None]).sum(axis=1)))
    assert not _golden_probs_ok()


def test_planted_onehot_sign_is_caught(monkeypatch):
    def bad(Z, lse, y, valid, coef):
        P = np.exp(Z - lse[:, None])
        rows = np.nonzero(valid)[0]
        P[rows, y[rows]] += 1.0
        P[~valid] = 0.0
        return P * coef
    monkeypatch.setattr(olc, "_dlogits", bad)
    with pytest.raises(AssertionError):
        test_finite_differences_flce()


def test_planted_transposed_grad_W_is_caught(monkeypatch):
    real = olc.flce_backward

    def bad(*a, **k):
        out = real(*a, **k)
        gW = out["grad_W"]
        out["grad_W"] = gW[::-1].copy()  # rows of grad_W swapped end for end
        return out
    monkeypatch.setattr(oracle, "flce_backward", bad)
    with pytest.raises(AssertionError):
        test_flce_matches_torch_autograd(False)


# ------------------------------------------ comparison metrics and the logits helper
#
# Every GPU gradient assertion goes through max_rel_err and normwise_err, and the
# invariant tests build dZ through flce_logits, so each is pinned here by values
# worked out by hand (the "derivation" comments), with a case that tells apart
# the plausible wrong versions: a denominator taken from `got`, a dropped abs,
# 0 returned for a zero reference, a max-row or spectral norm in place of the
# Frobenius norm, a dropped bias, a transposed weight, the wrong rows.

def _pin_max_rel(fn):
    # diff = [0, 0, -1] -> max|diff| = 1; max|ref| = 4 -> 0.25
    assert fn(np.array([1.0, 2.0, 3.0]), np.array([1.0, 2.0, 4.0])) == pytest.approx(0.25, abs=1e-15)
    # ref has its largest magnitude on a negative entry (-2): max|ref| = 2, not
    # max(ref) = 1; got - ref = [[-1, -0.5], [0, 0]] is never positive, so a
    # max without abs would give 0 -> 1 / 2 = 0.5
    assert fn(np.array([[-3.0, 0.0], [0.0, 1.0]]),
              np.array([[-2.0, 0.5], [0.0, 1.0]])) == pytest.approx(0.5, abs=1e-15)
    # the denominator is the reference's: max|got - ref| = 9, max|ref| = 1 -> 9
    assert fn(np.array([10.0, 0.0]), np.array([1.0, 0.0])) == pytest.approx(9.0, abs=1e-14)
    # zero reference: the absolute error, max|got| = 0.5 (0 would hide any error)
    assert fn(np.array([0.0, -0.5]), np.zeros(2)) == pytest.approx(0.5, abs=1e-15)
    assert fn(np.zeros((2, 3)), np.zeros((2, 3))) == 0.0
    # identical inputs, and bf16 torch tensors widened exactly: 1.5 and 3.0 are
    # bf16 values; |1.5 - 1.25| / 3 = 1/12
    t = torch.tensor([1.5, 3.0], dtype=torch.bfloat16)
    assert fn(t, t) == 0.0
    assert fn(t, np.array([1.25, 3.0])) == pytest.approx(1.0 / 12.0, abs=1e-15)


def _pin_normwise(fn):
    # ref = diag(3, 4): Frobenius norm 5 (spectral norm 4); got - ref = e_22:
    # norm 1 -> 1/5 = 0.2 (a spectral ratio would also give 1/4 = 0.25)
    ref = np.array([[3.0, 0.0], [0.0, 4.0]])
    assert fn(ref + np.array([[0.0, 0.0], [0.0, 1.0]]), ref) == pytest.approx(0.2, abs=1e-15)
    # the error spread over two rows: diff = [[0, 0.3], [0.4, 0]] -> 0.5 / 5 = 0.1
    # (a max-row norm would give 0.4 / 4 = 0.1 by accident here, so the next case)
    assert fn(ref + np.array([[0.0, 0.3], [0.4, 0.0]]), ref) == pytest.approx(0.1, abs=1e-15)
    # the whole error in one row: diff = [[0.6, 0.8], [0, 0]] -> 1 / 5 = 0.2
    # (max-row ratio 1 / 4 = 0.25)
    assert fn(ref + np.array([[0.6, 0.8], [0.0, 0.0]]), ref) == pytest.approx(0.2, abs=1e-15)
    # the denominator is the reference's: got = 2 ref -> ||ref|| / ||ref|| = 1
    # (dividing by ||got|| would give 1/2)
    assert fn(2.0 * ref, ref) == pytest.approx(1.0, abs=1e-15)
    # zero reference: the absolute norm, ||(3, 4)|| = 5
    assert fn(np.array([3.0, -4.0]), np.zeros(2)) == pytest.approx(5.0, abs=1e-15)
    assert fn(np.zeros(3), np.zeros(3)) == 0.0


def test_max_rel_err_hand_values():
    _pin_max_rel(oracle.max_rel_err)


def test_normwise_err_hand_values():
    _pin_normwise(oracle.normwise_err)


# H [3, 2], W [3, 2] (V = 3), bias [3]; the values of each case are worked out
# by hand in its comment.
_H = np.array([[1.0, 2.0], [3.0, -1.0], [0.0, 0.5]])
_W = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, -1.0]])
_B = np.array([0.5, -1.0, 0.0])


def _pin_flce_logits(fn):
    # row 2, h = (0, 0.5): h.w_v = (0, 0.5, -0.5); + bias -> (0.5, -0.5, -0.5)
    # row 0, h = (1, 2):   h.w_v = (1, 2, 0);      + bias -> (1.5, 1, 0)
    np.testing.assert_array_equal(fn(_H, _W, _B, np.array([2, 0])),
                                  [[0.5, -0.5, -0.5], [1.5, 1.0, 0.0]])
    # row 1, h = (3, -1), no bias: (3, -1, 7)
    np.testing.assert_array_equal(fn(_H, _W, None, np.array([1])), [[3.0, -1.0, 7.0]])
    # a non-square weight (V = 4, D = 2) and bf16 inputs widened exactly:
    # h = (2, 0.5): w = (1, 1), (-1, 0), (0, 4), (0.25, -2) -> (2.5, -2, 2, -0.5)
    W4 = torch.tensor([[1.0, 1.0], [-1.0, 0.0], [0.0, 4.0], [0.25, -2.0]], dtype=torch.bfloat16)
    H1 = torch.tensor([[2.0, 0.5]], dtype=torch.bfloat16)
    np.testing.assert_array_equal(fn(H1, W4, None, np.array([0])), [[2.5, -2.0, 2.0, -0.5]])


def test_flce_logits_hand_values():
    _pin_flce_logits(oracle.flce_logits)


def _fails(check, fn):
    try:
        check(fn)
    except (AssertionError, ValueError):
        return True
    return False


@pytest.mark.parametrize("bad", [
    lambda g, r: float(np.max(np.abs(olc._f64(g) - olc._f64(r))) / max(np.max(np.abs(olc._f64(g))), 1e-300)),
    lambda g, r: float(np.max(olc._f64(g) - olc._f64(r)) / np.max(np.abs(olc._f64(r))))
    if np.max(np.abs(olc._f64(r))) else 0.0,
    lambda g, r: float(np.max(np.abs(olc._f64(g) - olc._f64(r))) / np.max(olc._f64(r)))
    if np.max(olc._f64(r)) else 0.0,
    lambda g, r: float(np.max(np.abs(olc._f64(g) - olc._f64(r))) / np.max(np.abs(olc._f64(r))))
    if np.max(np.abs(olc._f64(r))) else 0.0,
], ids=["den_from_got", "no_abs_on_diff", "no_abs_on_ref", "zero_ref_gives_0"])
def test_planted_max_rel_err_mistakes_are_caught(bad):
    assert _fails(_pin_max_rel, bad)


@pytest.mark.parametrize("bad", [
    lambda g, r: float(np.linalg.norm(olc._f64(g) - olc._f64(r)) / np.linalg.norm(olc._f64(g)))
    if np.linalg.norm(olc._f64(g)) else 0.0,
    lambda g, r: float(np.linalg.norm(np.atleast_2d(olc._f64(g) - olc._f64(r)), 2) /
                       np.linalg.norm(np.atleast_2d(olc._f64(r)), 2))
    if np.linalg.norm(olc._f64(r)) else float(np.linalg.norm(olc._f64(g))),
    lambda g, r: float(np.max(np.linalg.norm(np.atleast_2d(olc._f64(g) - olc._f64(r)), axis=1)) /
                       np.max(np.linalg.norm(np.atleast_2d(olc._f64(r)), axis=1)))
    if np.linalg.norm(olc._f64(r)) else float(np.linalg.norm(olc._f64(g))),
    lambda g, r: float(np.linalg.norm(olc._f64(g) - olc._f64(r)) / np.linalg.norm(olc._f64(r)))
    if np.linalg.norm(olc._f64(r)) else 0.0,
], ids=["den_from_got", "spectral", "max_row_norm", "zero_ref_gives_0"])
def test_planted_normwise_err_mistakes_are_caught(bad):
    assert _fails(_pin_normwise, bad)


@pytest.mark.parametrize("bad", [
    lambda H, W, b, rows: olc._f64(H[rows]) @ olc._f64(W).T,                     # bias dropped
    lambda H, W, b, rows: olc._f64(H)[rows] @ olc._f64(W).T[:, ::-1] +
    (0 if b is None else olc._f64(b)),                                            # columns reversed
    lambda H, W, b, rows: olc._f64(H[np.sort(rows)]) @ olc._f64(W).T +
    (0 if b is None else olc._f64(b)),                                            # rows reordered
    lambda H, W, b, rows: (olc._f64(W) @ olc._f64(H[rows]).T).T[:, :olc._f64(W).shape[0]] * 1.0 +
    (0 if b is None else -olc._f64(b)),                                           # bias subtracted
], ids=["no_bias", "reversed_columns", "sorted_rows", "bias_sign"])
def test_planted_flce_logits_mistakes_are_caught(bad):
    assert _fails(_pin_flce_logits, bad)


def test_backward_with_forward_returns_the_forward():
    N, D, V = 33, 7, 301
    H, W, b, y = _rand(N, D, V, 41, ignore=(0, 9))
    rows = np.array([1, 4, 9, 30])
    for kw in ({}, {"rows": rows, "n_valid_total": N - 2}):
        gr = oracle.flce_backward(H, W, b, y, -100, "sum", 20, with_forward=True, **kw)
        f = oracle.flce_forward(H, W, b, y, -100, "sum", 20, rows=kw.get("rows"))
        for k in ("lse", "loss_rows", "label_logit"):
            np.testing.assert_array_equal(gr["forward"][k], f[k])
        assert gr["forward"]["loss"] == f["loss"] and gr["forward"]["n_valid"] == f["n_valid"]
        plain = oracle.flce_backward(H, W, b, y, -100, "sum", 20, **kw)
        for k in ("grad_H", "grad_W", "grad_b"):
            np.testing.assert_array_equal(gr[k], plain[k])


def _blockwise(blocks_got, blocks_ref):
    acc = oracle.BlockwiseError()
    for g, r in zip(blocks_got, blocks_ref):
        acc.add(g, r)
    return acc


def test_blockwise_error_hand_values():
    # ref = [[3, 0], [0, 4]] in two row blocks; got - ref = [[0, 0], [0, 1]]:
    # max|diff| = 1, max|ref| = 4 -> 0.25; ||diff|| = 1, ||ref|| = 5 -> 0.2
    acc = _blockwise([np.array([[3.0, 0.0]]), np.array([[0.0, 5.0]])],
                     [np.array([[3.0, 0.0]]), np.array([[0.0, 4.0]])])
    assert acc.max_rel() == pytest.approx(0.25, abs=1e-15)
    assert acc.normwise() == pytest.approx(0.2, abs=1e-15)
    # zero reference: the absolute errors, max 0.5 and norm sqrt(0.5^2 + 1.2^2) = 1.3
    acc = _blockwise([np.array([0.5]), np.array([-1.2])], [np.zeros(1), np.zeros(1)])
    assert acc.max_rel() == pytest.approx(1.2, abs=1e-15)
    assert acc.normwise() == pytest.approx(1.3, abs=1e-15)
    # an empty block changes nothing
    acc.add(np.zeros((0, 3)), np.zeros((0, 3)))
    assert acc.normwise() == pytest.approx(1.3, abs=1e-15)


def test_blockwise_error_equals_the_whole_tensor_functions():
    rng = np.random.default_rng(12)
    ref = rng.standard_normal((37, 11))
    got = ref + rng.standard_normal((37, 11)) * 1e-3
    acc = _blockwise([got[a:a + 8] for a in range(0, 37, 8)], [ref[a:a + 8] for a in range(0, 37, 8)])
    assert acc.max_rel() == pytest.approx(oracle.max_rel_err(got, ref), rel=1e-14)
    assert acc.normwise() == pytest.approx(oracle.normwise_err(got, ref), rel=1e-12)


_PACK_DOC = np.array([[1, 1, 1, 2, 2, 0, 0],
                      [1, 1, 1, 1, 1, 1, 1],
                      [0, 1, 2, 2, 2, 2, 2]])
# row 0: documents 1 (t 0-2) and 2 (t 3-4), then padding (t 5-6)
# row 1: one document over the whole row
# row 2: padding first (t 0), a one-token document (t 1), document 2 (t 2-6)
_PACK_WANT = np.array([[100, 101, -100, 103, -100, -100, -100],
                       [107, 108, 109, 110, 111, 112, -100],
                       [-100, -100, 116, 117, 118, 119, -100]])


def _check_packed(fn):
    y = np.arange(21).reshape(3, 7) + 100
    np.testing.assert_array_equal(fn(y, _PACK_DOC), _PACK_WANT)
    np.testing.assert_array_equal(y, np.arange(21).reshape(3, 7) + 100)  # input unchanged


def test_packed_document_labels_hand_values():
    _check_packed(oracle.packed_document_labels)
    y = np.arange(21).reshape(3, 7) + 100
    assert oracle.packed_document_labels(y, _PACK_DOC, ignore_index=-1)[0, 2] == -1


@pytest.mark.parametrize("bad", [
    lambda y, d: np.where(d == 0, -100, y),                                        # ends kept
    lambda y, d: np.where((d == 0) | (np.roll(d, 1, axis=1) != d), -100, y),       # first tokens
    lambda y, d: np.where(np.roll(d, -1, axis=1) != d, -100, y),                   # padding kept
], ids=["document_ends_kept", "first_tokens_dropped", "padding_kept"])
def test_planted_packed_label_mistakes_are_caught(bad):
    with pytest.raises(AssertionError):
        _check_packed(bad)
