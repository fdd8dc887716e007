"""fp64 CPU oracle of the language-model loss head.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import this module; the product path never does.  It shares no
code with the CUDA library and imports nothing from it.

What it computes is the plain definition of masked cross-entropy, which the
chunked methods on the source pages reach exactly (up to rounding order):

* Automodel PR #2996 "feat(loss): chunked masked CE, packing-mask preservation,
  scoped MoE AC", first commit message and "Proof": the chunked path computes the
  *identical* sum-reduced masked CE, checked against the full-tensor path and
  ``F.cross_entropy(reduction="sum")``; forward = per-row logsumexp + label-logit
  gather; backward = softmax recomputed, minus the one-hot label, times the
  incoming gradient; a ``num_label_tokens`` divisor with a guard for zero.
* Liger-Kernel issue #533 "Gradient checkpointing for grad_weight in LFCE",
  feature pitch: for fused linear CE the logits of a chunk are ``H_c @ W.T``,
  the gradient of the weight is accumulated as ``grad_W += dlogits_c.T @ H_c``
  (the ``addmm`` with beta=1) and the gradient of the input is
  ``dlogits_c @ W``.
* Liger-Kernel issue #941 "[Question] No gain in VRAM usage with
  LigerFusedLinearCrossEntropyLoss", model wiring: the weight is the
  ``[vocab, hidden]`` lm_head / tied-embedding matrix, the bias optional.

Every value is widened to float64 before any arithmetic.  The contractions use
numpy's ``@``; rows are processed in blocks only so that no float64 [N, V]
array is ever held (blocking does not change the definition: each row is
independent and the gradient sums are plain sums over rows).

Readings of points the pages leave open:

1. ``reduction="mean"`` divides by the number of non-ignored rows (the
   ``F.cross_entropy`` meaning).  If every row is ignored the loss and all
   gradients are 0 rather than 0/0.
2. A given ``num_label_tokens`` replaces the reduction's divisor; if it is 0 the
   loss and all gradients are 0 (the "zero num_label_tokens guard").
3. A label that is neither ``ignore_index`` nor in ``[0, V)`` is an error; the
   oracle raises ``ValueError`` for it.
4. The incoming gradient ``g`` of the scalar loss multiplies every gradient.
"""
from __future__ import annotations

import numpy as np

ROW_BLOCK = 512


# ----------------------------------------------------------------------------- helpers

def _f64(x):
    """Exact widening of an array-like (numpy or torch, bf16/fp32/fp64) to float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen in torch (numpy has no bf16)
        import torch
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def valid_rows(labels, V, ignore_index):
    """valid_i = (y_i != ignore_index); any other label outside [0, V) is an error."""
    y = _i64(labels)
    valid = y != ignore_index
    bad = valid & ((y < 0) | (y >= V))
    if bad.any():
        raise ValueError(f"label out of range at rows {np.nonzero(bad)[0][:8].tolist()}")
    return valid


def divisor(reduction, n_valid, num_label_tokens):
    """What the summed loss is divided by (readings 1 and 2 above)."""
    if num_label_tokens is not None:
        return int(num_label_tokens)
    if reduction == "sum":
        return 1
    if reduction == "mean":
        return int(n_valid)
    raise ValueError(f"unknown reduction {reduction!r}")


def scale(reduction, n_valid, num_label_tokens):
    """1/divisor, or 0 when the divisor is 0 (the zero guard)."""
    d = divisor(reduction, n_valid, num_label_tokens)
    return 0.0 if d == 0 else 1.0 / d


def logsumexp_rows(Z):
    """lse_i = m_i + log(sum_j exp(Z_ij - m_i)), m_i = max_j Z_ij."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def _blocks(N, block=ROW_BLOCK):
    for r0 in range(0, N, block):
        yield r0, min(N, r0 + block)


# ------------------------------------------------------------------ CE on given logits

def ce_forward(logits, labels, ignore_index=-100, reduction="sum", num_label_tokens=None):
    """Masked cross-entropy of given logits [N, V].

    Returns a dict with ``loss`` (float), ``n_valid`` (int), ``lse`` [N],
    ``loss_rows`` [N] (0 on ignored rows) and ``label_logit`` [N] (the gathered
    Z_{i, y_i}; NaN on ignored rows)."""
    N, V = logits.shape
    valid = valid_rows(labels, V, ignore_index)
    y = _i64(labels)
    lse = np.empty(N)
    zy = np.full(N, np.nan)
    for r0, r1 in _blocks(N):
        Z = _f64(logits[r0:r1])
        lse[r0:r1] = logsumexp_rows(Z)
        v = valid[r0:r1]
        rows = np.nonzero(v)[0]
        zy[r0 + rows] = Z[rows, y[r0 + rows]]
    return _finish_forward(lse, zy, valid, reduction, num_label_tokens)


def _finish_forward(lse, zy, valid, reduction, num_label_tokens):
    loss_rows = np.where(valid, lse - np.where(valid, zy, 0.0), 0.0)
    n_valid = int(valid.sum())
    S = float(np.sum(loss_rows))
    loss = S * scale(reduction, n_valid, num_label_tokens)
    return {"loss": loss, "sum": S, "n_valid": n_valid, "lse": lse,
            "loss_rows": loss_rows, "label_logit": zy}


def _dlogits(Z, lse, y, valid, coef):
    """dZ_ij = valid_i * (exp(Z_ij - lse_i) - [j == y_i]) * coef."""
    P = np.exp(Z - lse[:, None])
    rows = np.nonzero(valid)[0]
    P[rows, y[rows]] -= 1.0
    P[~valid] = 0.0
    return P * coef


def ce_backward(logits, labels, ignore_index=-100, reduction="sum", num_label_tokens=None,
                grad_loss=1.0, rows=None):
    """Gradient of the loss w.r.t. the given logits (float64 [N, V]).

    ``rows``, if given, restricts the output to those row indices (the scale
    still uses the count over all rows)."""
    N, V = logits.shape
    valid = valid_rows(labels, V, ignore_index)
    y = _i64(labels)
    coef = float(grad_loss) * scale(reduction, int(valid.sum()), num_label_tokens)
    idx = np.arange(N) if rows is None else np.asarray(rows)
    out = np.empty((len(idx), V))
    for b0, b1 in _blocks(len(idx)):
        r = idx[b0:b1]
        Z = _f64(logits[r])
        lse = logsumexp_rows(Z)
        out[b0:b1] = _dlogits(Z, lse, y[r], valid[r], coef)
    return out


# ------------------------------------------------------------- fused linear CE (FLCE)

def flce_logits(H, W, bias, rows):
    """Z = H[rows] @ W.T (+ bias), float64."""
    Z = _f64(H[rows]) @ _f64(W).T
    if bias is not None:
        Z += _f64(bias)[None, :]
    return Z


def flce_forward(H, W, bias, labels, ignore_index=-100, reduction="sum",
                 num_label_tokens=None, rows=None):
    """Forward of the fused linear CE: the masked CE of Z = H @ W.T + bias.

    ``rows`` restricts the per-row outputs to a subset (``loss`` is then the
    subset's sum times the scale computed from the subset's own count, so only
    the per-row fields are meaningful for a partial call)."""
    W64 = _f64(W)
    b64 = _f64(bias)
    V = W64.shape[0]
    y_all = _i64(labels)
    idx = np.arange(H.shape[0]) if rows is None else np.asarray(rows)
    valid_all = valid_rows(labels, V, ignore_index)
    valid = valid_all[idx]
    y = y_all[idx]
    lse = np.empty(len(idx))
    zy = np.full(len(idx), np.nan)
    for b0, b1 in _blocks(len(idx)):
        r = idx[b0:b1]
        Z = _f64(H[r]) @ W64.T
        if b64 is not None:
            Z += b64[None, :]
        lse[b0:b1] = logsumexp_rows(Z)
        v = np.nonzero(valid[b0:b1])[0]
        zy[b0 + v] = Z[v, y[b0 + v]]
    return _finish_forward(lse, zy, valid, reduction, num_label_tokens)


def flce_backward(H, W, bias, labels, ignore_index=-100, reduction="sum",
                  num_label_tokens=None, grad_loss=1.0, grad_W_init=None,
                  want_grad_H=True, want_grad_W=True, rows=None, n_valid_total=None,
                  with_forward=False):
    """Backward of the fused linear CE.

    grad_H = dZ @ W, grad_W = (grad_W_init or 0) + dZ.T @ H, grad_b = sum_i dZ_i,
    with dZ as in ``ce_backward``.  ``rows`` restricts the computation to a row
    subset; the scale then uses ``n_valid_total`` if given (the count over the
    whole problem), else the subset's own count.  ``with_forward`` also returns,
    under "forward", what ``flce_forward`` returns for the same rows (the
    backward forms the same logits and lse, so large problems need not form
    them twice)."""
    H64 = None
    W64 = _f64(W)
    b64 = _f64(bias)
    V, D = W64.shape
    N = H.shape[0]
    idx = np.arange(N) if rows is None else np.asarray(rows)
    valid_all = valid_rows(labels, V, ignore_index)
    y_all = _i64(labels)
    nv = int(valid_all[idx].sum()) if n_valid_total is None else int(n_valid_total)
    coef = float(grad_loss) * scale(reduction, nv, num_label_tokens)
    grad_H = np.zeros((len(idx), D)) if want_grad_H else None
    grad_W = (np.zeros((V, D)) if grad_W_init is None else _f64(grad_W_init).copy()) \
        if want_grad_W else None
    grad_b = np.zeros(V)
    lse_all = np.empty(len(idx))
    zy = np.full(len(idx), np.nan)
    for b0, b1 in _blocks(len(idx)):
        r = idx[b0:b1]
        H64 = _f64(H[r])
        Z = H64 @ W64.T
        if b64 is not None:
            Z += b64[None, :]
        lse = logsumexp_rows(Z)
        if with_forward:
            lse_all[b0:b1] = lse
            v = np.nonzero(valid_all[r])[0]
            zy[b0 + v] = Z[v, y_all[r][v]]
        dZ = _dlogits(Z, lse, y_all[r], valid_all[r], coef)
        if want_grad_H:
            grad_H[b0:b1] = dZ @ W64
        if want_grad_W:
            grad_W += dZ.T @ H64
        grad_b += dZ.sum(axis=0)
    out = {"grad_H": grad_H, "grad_W": grad_W, "grad_b": grad_b}
    if with_forward:
        out["forward"] = _finish_forward(lse_all, zy, valid_all[idx], reduction,
                                         num_label_tokens)
    return out


# ------------------------------------------------------------------ comparison metrics

def max_rel_err(got, ref):
    """max|got - ref| / max|ref| over the whole tensor (0 if both are 0)."""
    got = _f64(got)
    ref = _f64(ref)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def normwise_err(got, ref):
    """||got - ref||_F / ||ref||_F (absolute norm if ref is 0)."""
    got = _f64(got)
    ref = _f64(ref)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


class BlockwiseError:
    """max_rel_err and normwise_err of a tensor compared block by block (rows
    of a tensor too large to hold in float64 at once): the running
    max|got - ref|, max|ref|, sum (got - ref)^2 and sum ref^2 over the blocks
    give the same two numbers as the whole-tensor functions above."""

    def __init__(self):
        self.max_diff = 0.0
        self.max_ref = 0.0
        self.sq_diff = 0.0
        self.sq_ref = 0.0

    def add(self, got, ref):
        got = _f64(got)
        ref = _f64(ref)
        if ref.size == 0:
            return
        d = got - ref
        self.max_diff = max(self.max_diff, float(np.max(np.abs(d))))
        self.max_ref = max(self.max_ref, float(np.max(np.abs(ref))))
        self.sq_diff += float(np.sum(d * d))
        self.sq_ref += float(np.sum(ref * ref))

    def max_rel(self):
        return self.max_diff if self.max_ref == 0.0 else self.max_diff / self.max_ref

    def normwise(self):
        num = float(np.sqrt(self.sq_diff))
        den = float(np.sqrt(self.sq_ref))
        return num if den == 0.0 else num / den


# ----------------------------------------------------- packed-document label masking

def packed_document_labels(labels, doc_ids, ignore_index=-100):
    """Labels of packed sequences with the tokens that have no target ignored.

    Automodel PR #2996, "Summary" (packing-mask fix): an indexed packing mask
    holds 1, 2, ... for the packed documents of a row and 0 for padding.  A
    padding token has no label; neither has the last token of a document,
    whose next token starts another document (or the padding, or lies past
    the row).  labels and doc_ids are [B, T]; returns a new int64 [B, T]."""
    y = _i64(labels).copy()
    d = _i64(doc_ids)
    B, T = d.shape
    for r in range(B):
        for t in range(T):
            last = t == T - 1 or d[r, t + 1] != d[r, t]
            if d[r, t] == 0 or last:
                y[r, t] = ignore_index
    return y
