"""The data-parallel path on CPU: world_size-2 gloo ranks shard the rows,
exchange the valid-label count and the per-rank summed losses, and must
reproduce the single-process result.  The per-rank compute here is the fp64
oracle (the CUDA kernels need a GPU); what is under test is the sharding and
the exchange logic of lm_head_linear_fwd_gb300/dp.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _load_dp():
    # dp.py imports the package (which loads the CUDA library); on a CPU-only
    # machine load the module file with a stand-in for the library binding.
    import importlib.util
    import sys
    import types
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = types.ModuleType("_dp_pkg")
    pkg.__path__ = []
    sys.modules["_dp_pkg"] = pkg
    sys.modules["_dp_pkg._abi"] = types.ModuleType("_dp_pkg._abi")
    spec = importlib.util.spec_from_file_location(
        "_dp_pkg.dp", os.path.join(root, "lm_head_linear_fwd_gb300", "dp.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dp = _load_dp()
        rng = np.random.default_rng(0)
        N, D, V = 37, 6, 29
        H = rng.standard_normal((N, D))
        W = rng.standard_normal((V, D)) * 0.5
        y = rng.integers(0, V, N)
        y[[1, 7, 30]] = -100
        a, b = dp.shard_rows(N, rank, world)
        local = int((y[a:b] != -100).sum())
        total = int(dp.all_reduce_count(torch.tensor([local], dtype=torch.int64)).item())
        # each rank: its rows, divided by the global count
        f = oracle.flce_forward(H[a:b], W, None, y[a:b], -100, "sum", num_label_tokens=total)
        g = oracle.flce_backward(H[a:b], W, None, y[a:b], -100, "sum", num_label_tokens=total)
        gW = torch.tensor(g["grad_W"])
        dist.all_reduce(gW)  # the trainer's ordinary data-parallel gradient reduction
        s, n, mean = dp.combine_loss(torch.tensor(f["sum"], dtype=torch.float64),
                                      torch.tensor(f["n_valid"]))
        q.put((rank, total, f["loss"], s, n, mean, gW.numpy(), g["grad_H"], a, b))
    finally:
        dist.destroy_process_group()


def test_shard_rows_partition():
    dp = _load_dp()
    for N in (0, 1, 7, 64, 65537):
        for world in (1, 2, 3, 8):
            got = [dp.shard_rows(N, r, world) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == N
            assert all(got[i][1] == got[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in got]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_reproduce_the_global_mean():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    rng = np.random.default_rng(0)
    N, D, V = 37, 6, 29
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.5
    y = rng.integers(0, V, N)
    y[[1, 7, 30]] = -100
    ref = oracle.flce_forward(H, W, None, y, -100, "mean")
    refg = oracle.flce_backward(H, W, None, y, -100, "mean")
    assert all(r[1] == N - 3 for r in res)                       # global count on every rank
    assert sum(r[2] for r in res) == pytest.approx(ref["loss"], rel=1e-13)  # shares add up
    for r in res:
        assert r[4] == N - 3 and r[5] == pytest.approx(ref["loss"], rel=1e-13)
        np.testing.assert_allclose(r[6], refg["grad_W"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r[7], refg["grad_H"][r[8]:r[9]], rtol=1e-12, atol=1e-14)
