"""Scalar pure-Python restatement of the loss head for tiny inputs.

TEST INFRASTRUCTURE (see ``oracle/lm_head_ce.py``).  This is a second, loop-only
statement of the same definition, used to pin the numpy oracle: the logits are
formed by explicit dot products, the log-sum-exp is taken *without* the
max-subtraction (the textbook ``-log softmax`` gather), and every gradient is a
scalar loop.  Only for inputs small and well scaled enough that ``math.exp``
cannot overflow.
"""
from __future__ import annotations

import math


def logits(H, W, bias):
    N, D, V = len(H), len(H[0]), len(W)
    Z = [[0.0] * V for _ in range(N)]
    for i in range(N):
        for j in range(V):
            acc = 0.0
            for k in range(D):
                acc += float(H[i][k]) * float(W[j][k])
            if bias is not None:
                acc += float(bias[j])
            Z[i][j] = acc
    return Z


def ce(Z, labels, ignore_index, reduction, num_label_tokens, grad_loss=1.0):
    """Returns (loss, n_valid, dZ) for given logits Z (list of lists)."""
    N, V = len(Z), len(Z[0])
    n_valid = sum(1 for y in labels if y != ignore_index)
    if num_label_tokens is not None:
        div = num_label_tokens
    elif reduction == "sum":
        div = 1
    else:
        div = n_valid
    sc = 0.0 if div == 0 else 1.0 / div
    total = 0.0
    dZ = [[0.0] * V for _ in range(N)]
    for i in range(N):
        y = labels[i]
        if y == ignore_index:
            continue
        denom = 0.0
        for j in range(V):
            denom += math.exp(Z[i][j])
        total += -math.log(math.exp(Z[i][y]) / denom)
        for j in range(V):
            p = math.exp(Z[i][j]) / denom
            dZ[i][j] = (p - (1.0 if j == y else 0.0)) * grad_loss * sc
    return total * sc, n_valid, dZ


def flce(H, W, bias, labels, ignore_index, reduction, num_label_tokens, grad_loss=1.0):
    """Returns (loss, n_valid, grad_H, grad_W, grad_b), all from scalar loops."""
    Z = logits(H, W, bias)
    loss, n_valid, dZ = ce(Z, labels, ignore_index, reduction, num_label_tokens, grad_loss)
    N, D, V = len(H), len(H[0]), len(W)
    gH = [[0.0] * D for _ in range(N)]
    gW = [[0.0] * D for _ in range(V)]
    gb = [0.0] * V
    for i in range(N):
        for j in range(V):
            d = dZ[i][j]
            if d == 0.0:
                continue
            gb[j] += d
            for k in range(D):
                gH[i][k] += d * float(W[j][k])
                gW[j][k] += d * float(H[i][k])
    return loss, n_valid, gH, gW, gb
