"""Benchmark of the language-model loss head on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * fused linear CE forward + backward (logits = H W^T recomputed in the
    backward; grad_H, fp32 grad_W) on the chosen FLCE workload, default the
    Llama3-8B shape N=8192, D=4096, V=128256 bf16;
  * CE on given logits forward + in-place backward on [16384, 128256] bf16.
``value`` is the FLCE tokens/s of the step (the metric's first part); the
given-logits part is reported beside it (GB/s and its HBM roofline).

Timing: W warm-up steps, then exactly K timed steps between a barrier +
synchronize on both sides, CUDA events on the launching stream, max over
ranks.  Every input is larger than L2 (129 MB), so no flush is needed.
With --impl reference the fp64 CPU oracle is timed instead, on a bounded row
sample of the same workload, on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload llama3_8b_flce|long_packed_flce|small_flce]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per step, from
# in-limit ncu captures (one kernel, a few launches, a few GB resident) that
# are summarised under profiles/; each figure holds only for the kernel sources
# it was taken from (sha256 prefix of the listed files, comments left out) and
# is reported as null once the code of any of them changes.  CE on logits: the traffic of a [2048, 128256]
# capture scaled by the rows (every row is read, and written, once, so the
# traffic grows in proportion).  FLCE: the per-kernel captures of the
# benchmark's launches, summed over one step.
TRAFFIC = {
    # profiles/ce_logits_16384x128256_launch_list_and_small_case.md: 8 x the
    # 2048-row capture of the forward and the in-place backward
    "ce_logits": {"bytes_per_step": 12.12e9, "sha": "24b0a218c3d21127",
                  "files": ["ce_logits.cu", "common.cuh", "host.h"]},
    # profiles/flce_llama3_8b_kernel_traffic.md: the ten GEMM launches of one
    # step (forward; dZ, grad_H, grad_W of chunks of 3584, 3584 and 1024 rows)
    "flce": {"bytes_per_step": 33.85e9, "sha": "8b3a08a69a5b016c",
             "files": ["flce.cu", "tc_gemm.cuh", "common.cuh", "host.h"]},
}


def _code_only(text: bytes) -> bytes:
    """The source without its comments and blank lines: the hash follows the
    code the counters were taken on, not its commentary."""
    import re
    t = re.sub(rb"/\*.*?\*/", b" ", text, flags=re.S)
    t = re.sub(rb"//[^\n]*", b"", t)
    return b"\n".join(line.rstrip() for line in t.splitlines() if line.strip())


def csrc_sha(files=None):
    import glob
    import hashlib
    d = os.path.join(ROOT, "lm_head_linear_fwd_gb300", "csrc")
    if files is None:
        paths = sorted(glob.glob(os.path.join(d, "*.cu")) + glob.glob(os.path.join(d, "*.cuh")) +
                       glob.glob(os.path.join(d, "*.h")))
    else:
        paths = sorted(os.path.join(d, f) for f in files)
    h = hashlib.sha256()
    for f in paths:
        h.update(os.path.basename(f).encode())
        h.update(_code_only(open(f, "rb").read()))
    return h.hexdigest()[:16]


def traffic_for(part):
    t = TRAFFIC[part]
    if t["bytes_per_step"] is None or t["sha"] != csrc_sha(t["files"]):
        return None
    return t["bytes_per_step"]


METRIC = "tokens/s and % bf16 tensor peak for FLCE fwd+bwd; ce_logits HBM GB/s; peak extra GiB"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                if k in d and d[k]:
                    out[k] = float(d[k])
            if len(out) == 3:
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, ws, local
    return 0, 1, 0


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax.append(float(f[2]))
                except ValueError:
                    continue
                for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                    "sw_power_cap"), f[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def _events_time(fn, steps, stream, before=None):
    """Runs fn() `steps` times; returns per-step device ms (CUDA events on `stream`).
    `before()` (untimed) runs ahead of each step."""
    import torch
    times = []
    for _ in range(steps):
        if before is not None:
            before()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def run_ours(args, rank, ws, local):
    import torch
    import workloads as wl
    import lm_head_linear_fwd_gb300 as lh
    from lm_head_linear_fwd_gb300 import _abi

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    if args.only == "ce":
        return run_ce_only(args, rank, ws, local, dev, stream, peaks, peak_src)

    # ---------------------------------------------------------------- FLCE
    if args.tokens and args.workload == "llama3_8b_flce":
        p = wl.llama3_8b_flce(device=dev, N=args.tokens)
    elif args.tokens and args.workload == "long_packed_flce":
        p = wl.long_packed_flce(device=dev, B=1, T=args.tokens)
    else:
        p = wl.WORKLOADS[args.workload](device=dev)
    H, W, b, y = p.H, p.W, p.bias, p.labels
    N, D, V = p.N, p.D, p.V
    dt = _abi.FLCE_BF16 if H.dtype == torch.bfloat16 else _abi.FLCE_F32
    chunk = args.chunk or lh.flce_default_chunk(dt, N, D, V)
    torch.cuda.synchronize()
    base_mem = torch.cuda.memory_allocated(dev)
    ws_bytes = lh.flce_workspace_bytes(dt, N, D, V, chunk)
    wsbuf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = lh.new_status(dev)
    fo = lh.flce_fwd(H, W, y, b, p.ignore_index, p.reduction, p.num_label_tokens, ws=wsbuf,
                     status=status)
    one = torch.ones(1, device=dev)
    gH = torch.empty_like(H)
    gW = torch.empty((V, D), dtype=torch.float32, device=dev)
    gb = torch.empty(V, dtype=torch.float32, device=dev) if b is not None else None
    outputs_bytes = (gH.numel() * gH.element_size() + gW.numel() * 4 +
                     (gb.numel() * 4 if gb is not None else 0) + N * 4 + 16)

    def fwd():
        lh.flce_fwd(H, W, y, b, p.ignore_index, p.reduction, p.num_label_tokens, ws=wsbuf,
                    status=status, out=fo)

    def bwd():
        lh.flce_bwd(H, W, y, fo.lse, fo.n_valid, one, b, p.ignore_index, p.reduction,
                    p.num_label_tokens, chunk, grad_H=gH, grad_W=gW, grad_bias=gb, ws=wsbuf,
                    status=status)

    def step():
        fwd()
        bwd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    step()
    torch.cuda.synchronize()
    peak_extra = torch.cuda.max_memory_allocated(dev) - base_mem - outputs_bytes
    lh.check_status(status, "flce")

    fwd_ms = _events_time(fwd, max(1, min(args.steps, 3)), stream)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_host0 = time.perf_counter()
        step_ms = _events_time(step, args.steps, stream)
        torch.cuda.synchronize()
        host_s = time.perf_counter() - t_host0
    barrier(ws)
    clocks = clk.summary()
    flce_ms = max_over_ranks(sum(step_ms) / len(step_ms), ws)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    flops = 8.0 * N * D * V
    tflops = flops / (flce_ms * 1e-3) / 1e12
    tok_s = N * ws / (flce_ms * 1e-3)
    # the bias gradient's partial column sums come from the eight-warp dZ
    # epilogue (bf16, D <= 1024) or from one pass over dZ; grad_H's epilogue
    # warps add them up and grad_W's close a split-K grad_H, so neither takes
    # a launch of its own
    bias_kernels = 0 if b is None or (H.dtype == torch.bfloat16 and D <= 1024) else 1
    if chunk > 0:   # row chunks: dZ, grad_H, grad_W (+ the bias pass) per chunk
        n_chunks = (N + chunk - 1) // chunk
        launches_flce = 3 + n_chunks * (3 + bias_kernels)
        split = f"chunk={chunk}"
    else:           # vocabulary slices, then one rounding of the fp32 grad_H
        n_chunks = (V + (-chunk) - 1) // (-chunk)
        launches_flce = 3 + n_chunks * (3 + bias_kernels) + 1
        split = f"vocabulary slices of {-chunk} columns"
    if args.only == "flce-step":
        # profiling runs: the timed FLCE step alone, nothing else held on the device
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s",
                              "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": round(flce_ms, 4),
                              "config": {"workload": f"FLCE step only {args.workload} N={N} "
                                                     f"D={D} V={V}, {split}"},
                              "flce_tflops_8NDV": round(tflops, 2), "fwd_ms": round(fwd_avg, 4),
                              "peak_extra_gib": round(peak_extra / 2**30, 4), "clocks": clocks,
                              "note": "profiling run: FLCE step only"}))
        return

    # ------------------------------------- fused forward + backward (6NDV path)
    fws = torch.empty(int(_abi.flce_fwd_bwd_workspace_bytes(dt, N, D, V, chunk)),
                      dtype=torch.uint8, device=dev)
    del wsbuf
    torch.cuda.empty_cache()
    torch.cuda.synchronize()

    def fused():
        lh.flce_fwd_bwd(H, W, y, b, p.ignore_index, p.reduction, p.num_label_tokens, chunk, None,
                        ws=fws, status=status, grad_W=gW)

    fused()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    fused()
    torch.cuda.synchronize()
    fused_peak_extra = torch.cuda.max_memory_allocated(dev) - base_mem - outputs_bytes
    lh.check_status(status, "flce_fwd_bwd")
    fused_ms = max_over_ranks(sum(_events_time(fused, args.steps, stream)) / args.steps, ws)
    del fws
    torch.cuda.empty_cache()
    wsbuf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    # ------------------------------------------------------- e2e (host buffers)
    # Each step copies its inputs (H, W, labels, bias) from pinned host memory
    # and reads the loss back.  Pipelined as a training loop would: a copy
    # stream fills one of two device input sets while the other is computed.
    Hh = H.cpu().pin_memory()
    Wh = W.cpu().pin_memory()
    yh = y.cpu().pin_memory()
    bh = b.cpu().pin_memory() if b is not None else None
    n_e2e = max(2, args.steps)
    loss_h = torch.empty(n_e2e, dtype=torch.float32).pin_memory()
    sets = [(torch.empty_like(H), torch.empty_like(W), torch.empty_like(y),
             torch.empty_like(b) if b is not None else None) for _ in range(2)]
    copy_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def copy_in(k):
        Hd, Wd, yd, bd = sets[k]
        Hd.copy_(Hh, non_blocking=True)
        Wd.copy_(Wh, non_blocking=True)
        yd.copy_(yh, non_blocking=True)
        if bd is not None:
            bd.copy_(bh, non_blocking=True)

    def compute(k, i):
        Hd, Wd, yd, bd = sets[k]
        lh.flce_fwd(Hd, Wd, yd, bd, p.ignore_index, p.reduction, p.num_label_tokens, ws=wsbuf,
                    status=status, out=fo)
        lh.flce_bwd(Hd, Wd, yd, fo.lse, fo.n_valid, one, bd, p.ignore_index, p.reduction,
                    p.num_label_tokens, chunk, grad_H=gH, grad_W=gW, grad_bias=gb, ws=wsbuf,
                    status=status)
        loss_h[i].copy_(fo.loss[0], non_blocking=True)

    def e2e_pipelined(k_steps):
        with torch.cuda.stream(copy_stream):
            copy_in(0)
            ready[0].record(copy_stream)
        for i in range(k_steps):
            cur, nxt = i % 2, (i + 1) % 2
            if i + 1 < k_steps:
                with torch.cuda.stream(copy_stream):
                    if i >= 1:
                        copy_stream.wait_event(free[nxt])
                    copy_in(nxt)
                    ready[nxt].record(copy_stream)
            stream.wait_event(ready[cur])
            compute(cur, i)
            free[cur].record(stream)

    def e2e_serial(k_steps):
        for i in range(k_steps):
            copy_in(0)
            compute(0, i)

    def host_time(fn, k_steps):
        fn(2)
        torch.cuda.synchronize()
        barrier(ws)
        t0 = time.perf_counter()
        fn(k_steps)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e3 / k_steps

    e2e_ms = max_over_ranks(host_time(e2e_pipelined, n_e2e), ws)
    e2e_serial_ms = max_over_ranks(host_time(e2e_serial, n_e2e), ws)
    h2d = (H.numel() * H.element_size() + W.numel() * W.element_size() + y.numel() * 8 +
           (b.numel() * b.element_size() if b is not None else 0))
    del Hh, Wh, yh, bh, sets

    # ------------------------------------------- long-context packed workload
    long_line = None
    if args.only == "all":
        del H, W, b, y, gH, gW, gb, wsbuf, fo
        torch.cuda.empty_cache()
        q = wl.long_packed_flce(device=dev)
        qH, qW, qy = q.H, q.W, q.labels
        qc = lh.flce_default_chunk(dt, q.N, q.D, q.V)
        qws = torch.empty(lh.flce_workspace_bytes(dt, q.N, q.D, q.V, qc), dtype=torch.uint8,
                          device=dev)
        qgH = torch.empty_like(qH)
        qgW = torch.empty((q.V, q.D), dtype=torch.float32, device=dev)
        qfo = lh.flce_fwd(qH, qW, qy, None, q.ignore_index, q.reduction, q.num_label_tokens,
                          ws=qws, status=status)

        def qstep():
            lh.flce_fwd(qH, qW, qy, None, q.ignore_index, q.reduction, q.num_label_tokens,
                        ws=qws, status=status, out=qfo)
            lh.flce_bwd(qH, qW, qy, qfo.lse, qfo.n_valid, one, None, q.ignore_index,
                        q.reduction, q.num_label_tokens, qc, grad_H=qgH, grad_W=qgW, ws=qws,
                        status=status)

        for _ in range(2):
            qstep()
        torch.cuda.synchronize()
        qn = max(3, min(args.steps, 10))
        q_ms = max_over_ranks(sum(_events_time(qstep, qn, stream)) / qn, ws)
        lh.check_status(status, "long_packed_flce")
        q_tf = 8.0 * q.N * q.D * q.V / (q_ms * 1e-3) / 1e12
        long_line = {"workload": f"long_packed_flce N={q.N} D={q.D} V={q.V} bf16, chunk={qc}",
                     "ms": round(q_ms, 3), "tokens_per_s": round(q.N * ws / (q_ms * 1e-3), 1),
                     "tflops_8NDV": round(q_tf, 2),
                     "frac_of_peak": round(q_tf / peaks["bf16_tflops_sustained"], 4),
                     "steps": qn}
        del qH, qW, qy, qws, qgH, qgW, qfo, q
        torch.cuda.empty_cache()

    # free the FLCE buffers before the given-logits part
    if args.only != "all":
        del H, W, b, y, gH, gW, gb, wsbuf, fo
    del p
    torch.cuda.empty_cache()

    # ------------------------------------------------------ CE on given logits
    if args.only == "flce":
        line = {"metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(flce_ms, 4),
                "config": {"workload": f"FLCE only {args.workload} N={N} D={D} V={V}"},
                "flce_tflops_8NDV": round(tflops, 2), "clocks": clocks,
                "note": "profiling run: FLCE part only"}
        if rank == 0:
            print(json.dumps(line))
        return
    c = wl.ce_logits_large(device=dev, N=args.ce_rows)
    pristine = c.logits.clone()
    logits, labels = c.logits, c.labels
    cws = torch.empty(max(1, lh.ce_logits_workspace_bytes(c.N, c.V)), dtype=torch.uint8,
                      device=dev)
    cst = lh.new_status(dev)
    co = lh.ce_logits_fwd(logits, labels, c.ignore_index, c.reduction, c.num_label_tokens,
                          ws=cws, status=cst)

    def ce_step():
        lh.ce_logits_fwd(logits, labels, c.ignore_index, c.reduction, c.num_label_tokens,
                         ws=cws, status=cst, out=co)
        lh.ce_logits_bwd(logits, labels, co.lse, co.n_valid, one, c.ignore_index, c.reduction,
                         c.num_label_tokens, inplace_grad=True, status=cst)

    def restore():
        logits.copy_(pristine)

    for _ in range(args.warmup):
        restore()
        ce_step()
    torch.cuda.synchronize()
    base_ce = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    ce_step()
    torch.cuda.synchronize()
    ce_peak_extra = torch.cuda.max_memory_allocated(dev) - base_ce
    lh.check_status(cst, "ce_logits")
    barrier(ws)
    ce_times = _events_time(ce_step, args.steps, stream, before=restore)
    ce_ms = max_over_ranks(sum(ce_times) / len(ce_times), ws)
    ce_bytes = 3.0 * c.N * c.V * 2  # fwd read + bwd read + bwd write of the bf16 logits
    ce_N = c.N
    ce_gbs = ce_bytes / (ce_ms * 1e-3) / 1e9

    # the backward alone, with the saved lse and without it (out of place)
    restore()
    ce_bwd_line = ce_bwd_compare(c, co, cst, one, stream, args, ws, peaks)
    ce_one_line = ce_one_call(c, cst, stream, args, ws, peaks)
    del pristine, logits, c, cws, co
    torch.cuda.empty_cache()
    ce_odd_line = ce_odd_vocab(dev, stream, args, ws, peaks)

    # ------------------------------------------------- latency-bound workloads
    small = latency_configs(dev, stream, args.steps)

    # ------------------------------------------------------------ CPU baseline
    cpu = cpu_baseline(args) if (rank == 0 and not args.no_cpu_baseline) else None

    peak_t = peaks["bf16_tflops_sustained"]
    line = {
        "metric": METRIC,
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(flce_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the workload's shape)",
        "config": {
            "workload": (f"FLCE fwd+bwd {args.workload}: N={N} D={D} V={V} bf16, {split} "
                         "(value and ms_per_step); CE on given logits [16384,128256] bf16 "
                         "fwd + in-place bwd timed on its own (ce_logits)"),
            "global_batch": N * ws,
            "l2": "inputs larger than L2 (W and logits >= 1 GB); no flush",
            "parallelism": f"replicas x{ws} (tokens sharded, no collective)",
        },
        "flce": {
            "ms": round(flce_ms, 4),
            "fwd_ms": round(fwd_avg, 4),
            "tokens_per_s": round(tok_s, 1),
            "tflops_8NDV": round(tflops, 2),
            "mfu_6NDV_tflops": round(6.0 * N * D * V / (flce_ms * 1e-3) / 1e12, 2),
            "frac_of_peak": round(tflops / peak_t, 4),
            "peak_extra_gib": round(peak_extra / 2**30, 4),
            "bound_2048_row_fp32_tile_gib": round(2048 * V * 4 / 2**30, 4),
            "within_bound": bool(peak_extra <= 2048 * V * 4),
            "chunk": chunk,
        },
        "flce_fused_fwd_bwd": {
            "what": "flce_fwd_bwd: gradients formed in the forward, 6NDV flops",
            "ms": round(fused_ms, 4),
            "tokens_per_s": round(N * ws / (fused_ms * 1e-3), 1),
            "tflops_6NDV": round(6.0 * N * D * V / (fused_ms * 1e-3) / 1e12, 2),
            "frac_of_peak": round(6.0 * N * D * V / (fused_ms * 1e-3) / 1e12 / peak_t, 4),
            "peak_extra_gib": round(fused_peak_extra / 2**30, 4),
            "within_bound": bool(fused_peak_extra <= 2048 * V * 4),
        },
        "latency_workloads": small,
        "ce_logits": {
            "ms": round(ce_ms, 4),
            "gb_s": round(ce_gbs, 1),
            "frac_of_hbm": round(ce_gbs / peaks["hbm_gbs"], 4),
            "frac_of_8tbs": round(ce_gbs / 8000.0, 4),
            "peak_extra_gib": round(ce_peak_extra / 2**30, 6),
            "tokens_per_s": round(ce_N * ws / (ce_ms * 1e-3), 1),
            "bwd_only": ce_bwd_line,
            "fwd_bwd_one_call": ce_one_line,
            "odd_vocabulary": ce_odd_line,
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "tc_gemm_kernel (all four FLCE contractions), whole fwd+bwd step",
            "achieved": round(tflops, 2),
            "peak": peak_t,
            "unit": "TFLOP/s",
            "frac": round(tflops / peak_t, 4),
            "traffic": (traffic_for("flce")
                        if (args.workload == "llama3_8b_flce" and not args.tokens) else None),
            "traffic_unit": "bytes per step (all FLCE kernels, in-limit ncu captures)",
            "peak_source": f"bf16_tflops_sustained ({peak_src})",
        },
        "roofline_fwd": {
            "bound": "tensor",
            "kernel": "tc_gemm_kernel<EpiLse> + combine + finalize (flce_fwd)",
            "achieved": round(2.0 * N * D * V / (fwd_avg * 1e-3) / 1e12, 2),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(2.0 * N * D * V / (fwd_avg * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "peak_source": f"bf16_tflops burst ({peak_src})",
        },
        "roofline_ce_logits": {
            "bound": "hbm",
            "kernel": "ce_stream_kernel<fwd> + ce_stream_kernel<bwd> (+ finalize)",
            "achieved": round(ce_gbs, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(ce_gbs / peaks["hbm_gbs"], 4),
            "traffic": traffic_for("ce_logits") if args.ce_rows == 16384 else None,
            "traffic_unit": ("bytes per step (CE fwd + bwd kernels; a [2048, 128256] ncu "
                             "capture scaled by the rows)"),
            "peak_source": f"hbm_gbs ({peak_src})",
        },
        "e2e": {
            "value": round(N * ws / (e2e_ms * 1e-3), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": 4,
            "ms": round(e2e_ms, 4),
            "serial_ms": round(e2e_serial_ms, 4),
            "what": ("per step: pinned host H, W, labels -> device (copy stream, double-buffered "
                     "against the previous step's compute), flce_fwd + flce_bwd, loss -> host; "
                     "host wall time over the steps; serial_ms without the overlap"),
            "d2h_excludes": ("grad_H and the fp32 grad_W stay on the device (where an "
                             "optimizer step would use them); only the loss is read back"),
        },
        "long_packed_flce": long_line,
        "gpu_launches": int(args.steps * launches_flce),
        "clocks": clocks,
        "host_wall_s_timed": round(host_s, 3),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))


def ce_bwd_compare(c, co, cst, one, stream, args, ws, peaks):
    """Device time of the CE backward alone on the given-logits workload, with
    the forward's lse and without it (the row-cluster kernel), out of place."""
    import torch
    import lm_head_linear_fwd_gb300 as lh
    logits, labels = c.logits, c.labels
    gbuf = torch.empty_like(logits)
    n_valid_rows = int((labels != c.ignore_index).sum().item())

    def bwd(lse):
        return lambda: lh.ce_logits_bwd(logits, labels, lse, co.n_valid, one, c.ignore_index,
                                        c.reduction, c.num_label_tokens, grad_logits=gbuf,
                                        status=cst)
    bwd_ms = {}
    for name, fn in (("saved_lse", bwd(co.lse)), ("no_lse", bwd(None))):
        for _ in range(max(3, args.warmup)):
            fn()
        t = _events_time(fn, args.steps, stream)
        bwd_ms[name] = max_over_ranks(sum(t) / len(t), ws)
    lh.check_status(cst, "ce_logits_bwd")
    # the saved-lse kernel reads every row; the no-lse kernel skips ignored rows
    row_b = c.V * 2
    bwd_bytes = {"saved_lse": 2.0 * c.N * row_b,
                 "no_lse": (n_valid_rows + c.N) * float(row_b)}
    line = {name: {"ms": round(bwd_ms[name], 4),
                   "gb_s": round(bwd_bytes[name] / (bwd_ms[name] * 1e-3) / 1e9, 1),
                   "frac_of_hbm": round(bwd_bytes[name] / (bwd_ms[name] * 1e-3) / 1e9 /
                                        peaks["hbm_gbs"], 4)}
            for name in bwd_ms}
    line["bytes"] = ("saved_lse: read + write of every row; no_lse: read of the "
                     f"{n_valid_rows} non-ignored rows + write of all {c.N} rows "
                     "(a row cluster holds each row in shared memory: one read)")
    del gbuf
    return line


def ce_one_call(c, cst, stream, args, ws, peaks):
    """Device time of ce_logits_fwd_bwd (loss and gradient in one call, g = 1)
    on the given-logits workload, out of place, against the same bytes as the
    separate forward and in-place backward."""
    import torch
    import lm_head_linear_fwd_gb300 as lh
    logits, labels = c.logits, c.labels
    gbuf = torch.empty_like(logits)
    cws = torch.empty(max(1, lh.ce_logits_fwd_bwd_workspace_bytes(c.N, c.V)), dtype=torch.uint8,
                      device=logits.device)
    out, _ = lh.ce_logits_fwd_bwd(logits, labels, c.ignore_index, c.reduction,
                                  c.num_label_tokens, grad_logits=gbuf, ws=cws, status=cst)

    def fn():
        lh.ce_logits_fwd_bwd(logits, labels, c.ignore_index, c.reduction, c.num_label_tokens,
                             grad_logits=gbuf, ws=cws, status=cst, out=out)

    for _ in range(max(3, args.warmup)):
        fn()
    t = _events_time(fn, args.steps, stream)
    ms = max_over_ranks(sum(t) / len(t), ws)
    lh.check_status(cst, "ce_logits_fwd_bwd")
    n_valid_rows = int((labels != c.ignore_index).sum().item())
    nbytes = (n_valid_rows + c.N) * float(c.V * 2)
    del gbuf, cws
    return {"what": "ce_logits_fwd_bwd: loss and gradient in one call (g = 1), out of place",
            "ms": round(ms, 4),
            "tokens_per_s": round(c.N * ws / (ms * 1e-3), 1),
            "gb_s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "bytes": (f"read of the {n_valid_rows} non-ignored rows + write of all {c.N} rows "
                      "(a row cluster holds each row in shared memory)")}


def ce_odd_vocab(dev, stream, args, ws, peaks, V=50257):
    """CE on given logits with rows that start and end inside 16-byte blocks
    (an odd vocabulary, GPT-2's 50257): device time of the forward, the
    backward with the saved lse (out of place) and the one-call forward and
    backward, at the same 16384 rows."""
    import torch
    import workloads as wl
    import lm_head_linear_fwd_gb300 as lh
    c = wl.ce_logits_large(device=dev, N=args.ce_rows, V=V)
    x, y = c.logits, c.labels
    st = lh.new_status(dev)
    g = torch.ones(1, device=dev)
    gbuf = torch.empty_like(x)
    o = lh.ce_logits_fwd(x, y, c.ignore_index, c.reduction, status=st)
    fns = {
        "fwd": lambda: lh.ce_logits_fwd(x, y, c.ignore_index, c.reduction, status=st, out=o),
        "bwd_saved_lse": lambda: lh.ce_logits_bwd(x, y, o.lse, o.n_valid, g, c.ignore_index,
                                                  c.reduction, grad_logits=gbuf, status=st),
        "fwd_bwd_one_call": lambda: lh.ce_logits_fwd_bwd(x, y, c.ignore_index, c.reduction,
                                                         grad_logits=gbuf, status=st),
    }
    n_valid_rows = int((y != c.ignore_index).sum().item())
    row_b = float(V * 2)
    nbytes = {"fwd": c.N * row_b, "bwd_saved_lse": 2.0 * c.N * row_b,
              "fwd_bwd_one_call": (n_valid_rows + c.N) * row_b}
    line = {"what": f"CE on [{c.N}, {V}] bf16 logits: rows start and end inside 16-byte "
                    "blocks (partial first and last blocks)"}
    for name, fn in fns.items():
        for _ in range(max(3, args.warmup)):
            fn()
        t = _events_time(fn, args.steps, stream)
        ms = max_over_ranks(sum(t) / len(t), ws)
        gbs = nbytes[name] / (ms * 1e-3) / 1e9
        line[name] = {"ms": round(ms, 4), "gb_s": round(gbs, 1),
                      "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    lh.check_status(st, "ce_odd_vocab")
    del x, y, gbuf, o, c
    torch.cuda.empty_cache()
    return line


def run_ce_only(args, rank, ws, local, dev, stream, peaks, peak_src):
    """Given-logits part alone (profiling runs)."""
    import torch
    import workloads as wl
    import lm_head_linear_fwd_gb300 as lh
    c = wl.ce_logits_large(device=dev, N=args.ce_rows)
    logits, labels = c.logits, c.labels
    cws = torch.empty(max(1, lh.ce_logits_workspace_bytes(c.N, c.V)), dtype=torch.uint8,
                      device=dev)
    cst = lh.new_status(dev)
    one = torch.ones(1, device=dev)
    co = lh.ce_logits_fwd(logits, labels, c.ignore_index, c.reduction, ws=cws, status=cst)

    def ce_step():
        lh.ce_logits_fwd(logits, labels, c.ignore_index, c.reduction, ws=cws, status=cst, out=co)
        lh.ce_logits_bwd(logits, labels, co.lse, co.n_valid, one, c.ignore_index, c.reduction,
                         inplace_grad=True, status=cst)

    for _ in range(args.warmup):
        ce_step()
    t = _events_time(ce_step, args.steps, stream)
    ms = max_over_ranks(sum(t) / len(t), ws)
    gbs = 3.0 * c.N * c.V * 2 / (ms * 1e-3) / 1e9
    bwd_line = ce_bwd_compare(c, co, cst, one, stream, args, ws, peaks)
    one_line = ce_one_call(c, cst, stream, args, ws, peaks)
    N, V = c.N, c.V
    del c, logits, labels, cws, co
    torch.cuda.empty_cache()
    odd_line = ce_odd_vocab(dev, stream, args, ws, peaks)
    if rank == 0:
        print(json.dumps({"metric": METRIC, "value": round(gbs, 1), "unit": "GB/s",
                          "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": round(ms, 4),
                          "config": {"workload": f"CE on logits only [{N},{V}] bf16"},
                          "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                          "bwd_only": bwd_line,
                          "fwd_bwd_one_call": one_line,
                          "odd_vocabulary": odd_line,
                          "note": "profiling run: given-logits part only"}))


def latency_configs(dev, stream, steps):
    """fwd+bwd of the two small FLCE workloads (tiny fp32; the small bf16 model
    with bias), launched eagerly and replayed from a CUDA graph."""
    import torch
    import workloads as wl
    import lm_head_linear_fwd_gb300 as lh
    out = {}
    for name, p in (("tiny_flce N=256 D=128 V=1000 fp32", wl.tiny_flce(device=dev)),
                    ("small_flce N=2048 D=768 V=32777 bf16+bias", wl.small_flce(device=dev))):
        H, W, b, y = p.H, p.W, p.bias, p.labels
        N, D, V = p.N, p.D, p.V
        dt = 0 if H.dtype == torch.bfloat16 else 1
        ws = torch.empty(lh.flce_workspace_bytes(dt, N, D, V, 0), dtype=torch.uint8, device=dev)
        st = lh.new_status(dev)
        one = torch.ones(1, device=dev)
        gH = torch.empty_like(H)
        gW = torch.empty(V, D, device=dev)
        gb = torch.empty(V, device=dev) if b is not None else None
        fo = lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, ws=ws, status=st)

        def step():
            lh.flce_fwd(H, W, y, b, -100, p.reduction, p.num_label_tokens, ws=ws, status=st,
                        out=fo)
            lh.flce_bwd(H, W, y, fo.lse, fo.n_valid, one, b, -100, p.reduction,
                        p.num_label_tokens, None, grad_H=gH, grad_W=gW, grad_bias=gb, ws=ws,
                        status=st)

        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        eager = sum(_events_time(step, steps, stream)) / steps
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        graph = sum(_events_time(g.replay, steps, stream)) / steps
        lh.check_status(st)
        out[name] = {"eager_ms": round(eager, 4), "graph_ms": round(graph, 4),
                     "tokens_per_s_graph": round(N / (graph * 1e-3), 1),
                     "tflops_8NDV_graph": round(8.0 * N * D * V / (graph * 1e-3) / 1e12, 2)}
    return out


# ------------------------------------------------------------- oracle timing

def blas_info():
    """Name and thread count of the BLAS numpy (and so the oracle) runs on."""
    import ctypes
    import glob
    import numpy as np
    name = None
    try:
        name = np.show_config(mode="dicts")["Build Dependencies"]["blas"]["name"]
    except Exception:
        pass
    try:
        import threadpoolctl
        for d in threadpoolctl.threadpool_info():
            if d.get("user_api") == "blas":
                return {"name": d.get("internal_api") or name, "threads": d.get("num_threads")}
    except ImportError:
        pass
    libdir = os.path.join(os.path.dirname(np.__file__), os.pardir, "numpy.libs")
    for path in glob.glob(os.path.join(libdir, "*openblas*.so*")):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                    "openblas_get_num_threads64_", "openblas_get_num_threads"):
            f = getattr(lib, sym, None)
            if f is not None:
                return {"name": name, "threads": int(f())}
    return {"name": name, "threads": None}


def cpu_baseline(args, rows=None, workload=None):
    """The fp64 oracle (as it stands) on a bounded row sample of the FLCE workload."""
    import numpy as np

    import oracle
    import workloads as wl
    wname = workload or args.workload
    rows = rows or args.cpu_rows
    p = wl.WORKLOADS[wname](device="cpu") if wname != "long_packed_flce" else \
        wl.long_packed_flce(device="cpu")
    rng = np.random.default_rng(0)
    sel = np.sort(rng.choice(p.N, rows, replace=False))
    t0 = time.perf_counter()
    oracle.flce_forward(p.H, p.W, p.bias, p.labels, p.ignore_index, p.reduction,
                        p.num_label_tokens, rows=sel)
    oracle.flce_backward(p.H, p.W, p.bias, p.labels, p.ignore_index, p.reduction,
                         p.num_label_tokens, rows=sel)
    dt = time.perf_counter() - t0
    blas = blas_info()
    return {"value": round(rows / dt, 3), "unit": "tokens/s",
            "cores": blas["threads"] or os.cpu_count(), "host_cores": os.cpu_count(),
            "blas": blas, "kind": "oracle",
            "sample": f"{rows} sampled rows of {wname} (N={p.N}, D={p.D}, V={p.V}), fwd+bwd in "
                      f"fp64 numpy, {dt:.2f} s"}


def run_reference(args, rank, ws):
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads as wl
    p = wl.WORKLOADS[args.workload](device="cpu")
    rng = np.random.default_rng(0)
    rows = args.cpu_rows
    times = []
    for i in range(args.warmup + args.steps):
        sel = np.sort(rng.choice(p.N, rows, replace=False))
        t0 = time.perf_counter()
        oracle.flce_forward(p.H, p.W, p.bias, p.labels, p.ignore_index, p.reduction,
                            p.num_label_tokens, rows=sel)
        oracle.flce_backward(p.H, p.W, p.bias, p.labels, p.ignore_index, p.reduction,
                             p.num_label_tokens, rows=sel)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    v = rows / per
    blas = blas_info()
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 3),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"FLCE fwd+bwd {args.workload}: N={p.N} D={p.D} V={p.V}; each "
                               f"step a {rows}-row sample",
                   "global_batch": rows, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s",
                         "cores": blas["threads"] or os.cpu_count(), "host_cores": os.cpu_count(),
                         "blas": blas, "kind": "oracle",
                         "sample": f"{rows} rows per step of {args.workload}"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_flce",
                    choices=["llama3_8b_flce", "long_packed_flce", "small_flce"])
    ap.add_argument("--cpu-rows", type=int, default=32)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override N of the FLCE workload (smaller cases for profiling)")
    ap.add_argument("--only", choices=["all", "flce", "flce-step", "ce"], default="all",
                    help="run one part only (profiling runs)")
    ap.add_argument("--chunk", type=int, default=0,
                    help="FLCE backward split: rows per chunk, or minus the columns of each "
                         "vocabulary slice (default: the library's row chunk)")
    ap.add_argument("--ce-rows", type=int, default=16384,
                    help="rows of the given-logits workload (smaller cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, ws, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, ws)
    else:
        run_ours(args, rank, ws, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
