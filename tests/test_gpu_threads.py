"""The library is called from threads that have only used the CUDA runtime
lazily (autograd runs the backward on its own device thread)."""
import threading

import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def test_flce_from_a_fresh_thread():
    import lm_head_linear_fwd_gb300 as lh
    p = wl.random_flce(300, 128, 1000, torch.bfloat16, bias=True, seed=5, reduction="mean")
    H, W, b, y = p.H.cuda(), p.W.cuda(), p.bias.cuda(), p.labels.cuda()
    box = {}

    def work():
        try:
            out = lh.flce_fwd(H, W, y, b, -100, "mean")
            bw = lh.flce_bwd(H, W, y, out.lse, out.n_valid, torch.ones(1, device="cuda"), b, -100,
                             "mean", None, 256)
            torch.cuda.synchronize()
            box["out"], box["bw"] = out, bw
        except Exception as e:  # surfaced in the main thread
            box["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in box, box.get("err")
    ref = oracle.flce_forward(p.H, p.W, p.bias, p.labels, -100, "mean")
    assert abs(box["out"].loss.item() - ref["loss"]) <= 1e-3 * ref["loss"]
    gr = oracle.flce_backward(p.H, p.W, p.bias, p.labels, -100, "mean")
    assert oracle.max_rel_err(box["bw"].grad_W.cpu(), gr["grad_W"]) <= 2e-2
