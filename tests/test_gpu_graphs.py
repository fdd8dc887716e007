"""Both operations captured in a CUDA graph: replays give the eager results
bit for bit (the library only enqueues work on the caller's stream once each
kernel has run once on the device)."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def test_flce_and_ce_in_a_cuda_graph():
    import lm_head_linear_fwd_gb300 as lh
    p = wl.random_flce(1000, 256, 5000, torch.bfloat16, bias=True, seed=31, reduction="mean")
    H, W, b, y = p.H.cuda(), p.W.cuda(), p.bias.cuda(), p.labels.cuda()
    c = wl.random_ce(512, 7000, torch.bfloat16, seed=32)
    logits0 = c.logits.cuda().contiguous()
    logits = logits0.clone()
    yl = c.labels.cuda()
    N, D, V = p.N, p.D, p.V
    ws = torch.empty(lh.flce_workspace_bytes(0, N, D, V, 256), dtype=torch.uint8, device="cuda")
    st = lh.new_status("cuda")
    one = torch.ones(1, device="cuda")
    gH = torch.empty_like(H)
    gW = torch.empty(V, D, device="cuda")
    gb = torch.empty(V, device="cuda")
    fo = lh.flce_fwd(H, W, y, b, -100, "mean", ws=ws, status=st)
    co = lh.ce_logits_fwd(logits, yl, status=st)

    def step():
        lh.flce_fwd(H, W, y, b, -100, "mean", ws=ws, status=st, out=fo)
        lh.flce_bwd(H, W, y, fo.lse, fo.n_valid, one, b, -100, "mean", None, 256, grad_H=gH,
                    grad_W=gW, grad_bias=gb, ws=ws, status=st)
        logits.copy_(logits0)
        lh.ce_logits_fwd(logits, yl, status=st, out=co)
        lh.ce_logits_bwd(logits, yl, co.lse, co.n_valid, one, inplace_grad=True, status=st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()   # eager, on the capture stream: every kernel has run once
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (fo.loss, fo.lse, gH, gW, gb, co.loss, logits)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (gH, gW, gb):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        lh.check_status(st)
        for a, e in zip((fo.loss, fo.lse, gH, gW, gb, co.loss, logits), eager):
            assert torch.equal(a, e)


def test_ce_without_saved_lse_in_a_cuda_graph():
    # the row-cluster backward (a cluster launch) and the unaligned-row
    # fallback, each captured after one eager run
    import lm_head_linear_fwd_gb300 as lh
    cases = [wl.random_ce(96, 128256, torch.bfloat16, seed=41),
             wl.random_ce(64, 1003, torch.bfloat16, seed=42)]
    dev = [(c.logits.cuda().contiguous(), c.labels.cuda()) for c in cases]
    st = lh.new_status("cuda")
    one = torch.ones(1, device="cuda")
    outs = [lh.ce_logits_fwd(x, y, reduction="mean", status=st) for x, y in dev]
    grads = [torch.empty_like(x) for x, _ in dev]

    def step():
        for (x, y), o, g in zip(dev, outs, grads):
            lh.ce_logits_fwd(x, y, reduction="mean", status=st, out=o)
            lh.ce_logits_bwd(x, y, None, o.n_valid, one, reduction="mean", grad_logits=g,
                             status=st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [g.clone() for g in grads]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for g in grads:
            g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        lh.check_status(st)
        for g, e in zip(grads, eager):
            assert torch.equal(g, e)


def test_ce_fwd_bwd_in_a_cuda_graph():
    # the one-call forward and backward: the row-cluster kernel in its fused
    # mode, and the two-call fallback for unaligned rows
    import lm_head_linear_fwd_gb300 as lh
    cases = [wl.random_ce(96, 128256, torch.bfloat16, seed=43),
             wl.random_ce(64, 1003, torch.bfloat16, seed=44)]
    dev = [(c.logits.cuda().contiguous(), c.labels.cuda()) for c in cases]
    st = lh.new_status("cuda")
    half = torch.full((1,), 0.5, device="cuda")
    grads = [torch.empty_like(x) for x, _ in dev]
    outs = [lh.ce_logits_fwd_bwd(x, y, reduction="mean", grad_loss=half, grad_logits=g,
                                 want_lse=True, status=st)[0]
            for (x, y), g in zip(dev, grads)]

    def step():
        for (x, y), o, g in zip(dev, outs, grads):
            lh.ce_logits_fwd_bwd(x, y, reduction="mean", grad_loss=half, grad_logits=g,
                                 status=st, out=o)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    res = lambda: [t for o, g in zip(outs, grads) for t in (o.loss, o.lse.nan_to_num(0.0), g)]
    eager = [t.clone() for t in res()]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for o, g in zip(outs, grads):
            g.zero_()
            o.loss.zero_()
        graph.replay()
        torch.cuda.synchronize()
        lh.check_status(st)
        for a, e in zip(res(), eager):
            assert torch.equal(a, e)
