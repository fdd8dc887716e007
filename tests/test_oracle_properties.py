"""Property-based pin of the fp64 oracle against the loop-only restatement
(oracle/bruteforce.py) over random tiny problems: shapes down to one row,
one feature and one class, with and without bias, ignored rows, an
ignore_index inside the vocabulary, every reduction, num_label_tokens given
(zero included) or not, and any incoming gradient.  Both sides must agree to
rounding (the restatement takes exp without the max-subtraction, so logits
are kept small)."""
import numpy as np
import pytest

import oracle
from oracle import bruteforce

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def problems(draw):
    N = draw(st.integers(1, 6))
    D = draw(st.integers(1, 5))
    V = draw(st.integers(1, 9))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.7
    b = rng.standard_normal(V) * 0.3 if draw(st.booleans()) else None
    ignore_index = draw(st.sampled_from([-100, 0, V - 1]))
    y = rng.integers(0, V, N)
    mask = rng.random(N) < draw(st.sampled_from([0.0, 0.3, 1.0]))
    y[mask] = ignore_index
    reduction = draw(st.sampled_from(["sum", "mean"]))
    nlt = draw(st.sampled_from([None, 0, 1, 7]))
    g = draw(st.sampled_from([1.0, 0.5, -2.0, 0.0]))
    return H, W, b, y, ignore_index, reduction, nlt, g


@hypothesis.settings(max_examples=80, deadline=None)
@hypothesis.given(problems())
def test_oracle_matches_loop_restatement(prob):
    H, W, b, y, ig, reduction, nlt, g = prob
    loss, nv, gH, gW, gb = bruteforce.flce(H.tolist(), W.tolist(),
                                           None if b is None else b.tolist(), y.tolist(), ig,
                                           reduction, nlt, grad_loss=g)
    f = oracle.flce_forward(H, W, b, y, ig, reduction, nlt)
    gr = oracle.flce_backward(H, W, b, y, ig, reduction, nlt, grad_loss=g)
    assert f["n_valid"] == nv
    assert f["loss"] == pytest.approx(loss, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(gr["grad_H"], gH, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(gr["grad_W"], gW, rtol=1e-11, atol=1e-13)
    if b is not None:
        np.testing.assert_allclose(gr["grad_b"], gb, rtol=1e-11, atol=1e-13)
    # given logits: the CE part alone against the same restatement
    Z = H @ W.T + (0.0 if b is None else b)
    closs, cnv, dZ = bruteforce.ce(Z.tolist(), y.tolist(), ig, reduction, nlt, grad_loss=g)
    cf = oracle.ce_forward(Z, y, ig, reduction, nlt)
    assert cf["n_valid"] == cnv
    assert cf["loss"] == pytest.approx(closs, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(oracle.ce_backward(Z, y, ig, reduction, nlt, grad_loss=g), dZ,
                               rtol=1e-11, atol=1e-13)
