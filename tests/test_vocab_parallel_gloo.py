"""The vocabulary-parallel exchange on CPU: two gloo ranks each own half of the
vocabulary and run lm_head_linear_fwd_gb300.vocab_parallel.forward/backward
with per-shard steps written here in float64 (the CUDA kernels need a GPU);
what is under test is the order of phases and collectives of the module."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

N, D, V, SPLIT = 29, 5, 23, 11
LOG2E = 1.0 / math.log(2.0)


def _data():
    rng = np.random.default_rng(4)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.7
    b = rng.standard_normal(V) * 0.2
    y = rng.integers(0, V, N)
    y[[2, 9]] = -100
    y[0], y[1] = SPLIT - 1, SPLIT  # both sides of the shard edge
    return H, W, b, y


class Float64ShardOps:
    """Per-shard steps restated in float64 numpy (stand-ins for the kernels)."""

    def partials(self, H, W, labels, v0, V_total, bias, ignore_index, status):
        Z = H.numpy() @ W.numpy().T + bias.numpy()
        t = Z * LOG2E
        m = t.max(axis=1)
        s = np.exp2(t - m[:, None]).sum(axis=1)
        y = labels.numpy()
        inside = (y != ignore_index) & (y >= v0) & (y < v0 + W.shape[0])
        zy = np.where(inside, Z[np.arange(len(y)), np.clip(y - v0, 0, W.shape[0] - 1)], 0.0)
        return torch.tensor(m), torch.tensor(s), torch.tensor(zy)

    def rescale(self, m, s, m_global):
        return s * torch.exp2(m - m_global)

    def finish(self, m_g, s_g, zy_g, labels, V_total, ignore_index, reduction, nlt, status):
        lse = (m_g + torch.log2(s_g)) / LOG2E
        valid = labels != ignore_index
        rows = torch.where(valid, lse - zy_g, torch.zeros_like(lse))
        n = int(valid.sum())
        div = n if reduction == "mean" else 1
        return (lse, torch.tensor([float(rows.sum()) / div], dtype=torch.float64),
                torch.tensor([n]))

    def backward(self, H, W, labels, v0, V_total, bias, ignore_index, reduction, nlt, lse,
                 n_valid, grad_loss, chunk, want_H, want_W, status):
        Z = H.numpy() @ W.numpy().T + bias.numpy()
        P = np.exp(Z - lse.numpy()[:, None])
        y = labels.numpy()
        valid = y != ignore_index
        for i in np.nonzero(valid & (y >= v0) & (y < v0 + W.shape[0]))[0]:
            P[i, y[i] - v0] -= 1.0
        P[~valid] = 0.0
        coef = float(grad_loss) / (int(n_valid) if reduction == "mean" else 1)
        dZ = P * coef
        return (torch.tensor(dZ @ W.numpy()), torch.tensor(dZ.T @ H.numpy()),
                torch.tensor(dZ.sum(axis=0)))


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        from lm_head_linear_fwd_gb300 import vocab_parallel as vp
        H, W, b, y = _data()
        a, c = (0, SPLIT) if rank == 0 else (SPLIT, V)
        Ht, yt = torch.tensor(H), torch.tensor(y)
        f = vp.forward(Ht, torch.tensor(W[a:c]), yt, a, V, torch.tensor(b[a:c]),
                       reduction="mean", ops=Float64ShardOps(), status=torch.zeros(1))
        gH, gW, gb = vp.backward(Ht, torch.tensor(W[a:c]), yt, a, V, f, torch.tensor(1.0),
                                 torch.tensor(b[a:c]), reduction="mean", ops=Float64ShardOps())
        q.put((rank, float(f.loss), f.lse.numpy(), gH.numpy(), gW.numpy(), gb.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reproduce_the_unsharded_oracle():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=240) for _ in range(2)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    H, W, b, y = _data()
    ref = oracle.flce_forward(H, W, b, y, -100, "mean")
    gr = oracle.flce_backward(H, W, b, y, -100, "mean")
    for r in res:
        assert r[1] == pytest.approx(ref["loss"], rel=1e-12)
        np.testing.assert_allclose(r[2], ref["lse"], rtol=1e-12)
        np.testing.assert_allclose(r[3], gr["grad_H"], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(np.concatenate([res[0][4], res[1][4]]), gr["grad_W"], rtol=1e-10,
                               atol=1e-13)
    np.testing.assert_allclose(np.concatenate([res[0][5], res[1][5]]), gr["grad_b"], rtol=1e-10,
                               atol=1e-13)
