"""Seeded synthetic inputs for the language-model loss head.

This module only draws random numbers and lays them out; it holds none of the
loss head's arithmetic.  Both the CUDA path (tests, benchmark) and the fp64 CPU
oracle take their inputs from here, so they see the same bytes.

The workloads stand in for the ones on the source pages:

* ``tiny_flce``        N=256, D=128, V=1000, fp32 (a case the oracle finishes in
                       well under a second).
* ``ce_logits_large``  given logits [16384, 128256] bf16 ~ N(0, 2): the shape
                       Automodel PR #2996 quotes its memory numbers on (its
                       ChunkedCrossEntropy commit message).
* ``small_flce``       B=2, T=1024, D=768, V=32777 with bias: the small model of
                       Liger-Kernel issue #941 (hidden 768, vocab 32777).
* ``llama3_8b_flce``   N=8192, D=4096, V=128256: the Llama3-8B shape of
                       torchtitan PR #996.
* ``long_packed_flce`` B=4 rows of T=16384 tokens, 4 packed documents per row,
                       D=5120, V=151936, padding tail and document boundaries
                       ignored (the long-context packed case of Automodel PR
                       #2996, "Motivation").

Values are drawn in fp32 with ``torch`` generators seeded per workload, then
rounded once (round-to-nearest-even) to bf16 where the workload is bf16.
Large tensors can be drawn directly on a CUDA device; the draw is deterministic
for a given device type, seed and shape, and a test that needs the oracle copies
the exact bytes back to the host.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass
class FLCEInputs:
    """Inputs of the fused linear cross-entropy: logits = H @ W.T (+ bias)."""
    name: str
    H: torch.Tensor            # [N, D]
    W: torch.Tensor            # [V, D] (tied-embedding layout)
    bias: Optional[torch.Tensor]  # [V] or None
    labels: torch.Tensor       # [N] int64
    ignore_index: int
    reduction: str             # "sum" or "mean"
    num_label_tokens: Optional[int]

    @property
    def N(self):
        return self.H.shape[0]

    @property
    def D(self):
        return self.H.shape[1]

    @property
    def V(self):
        return self.W.shape[0]


@dataclasses.dataclass
class CEInputs:
    """Inputs of the cross-entropy on given logits."""
    name: str
    logits: torch.Tensor       # [N, V]
    labels: torch.Tensor       # [N] int64
    ignore_index: int
    reduction: str
    num_label_tokens: Optional[int]
    inplace_grad: bool

    @property
    def N(self):
        return self.logits.shape[0]

    @property
    def V(self):
        return self.logits.shape[1]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device).type)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, dtype: torch.dtype, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, then rounded once to ``dtype``."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform_labels(N: int, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(0, V, (N,), generator=g, device=device, dtype=torch.int64)


def zipf_labels(N: int, V: int, s: float, seed: int, device="cpu") -> torch.Tensor:
    """Ids k in [0, V) with P(k) proportional to (k+1)^-s, by inverse-CDF sampling."""
    k = torch.arange(1, V + 1, dtype=torch.float64)
    cdf = torch.cumsum(k.pow(-s), 0)
    cdf /= cdf[-1].clone()
    g = _gen(seed, "cpu")
    u = torch.rand(N, generator=g, dtype=torch.float64)
    ids = torch.searchsorted(cdf, u, right=True).clamp_(max=V - 1)
    return ids.to(device=device, dtype=torch.int64)


def mask_fraction(labels: torch.Tensor, frac: float, seed: int, ignore_index=IGNORE_INDEX) -> int:
    """Set round(frac*N) distinct positions (seeded permutation) to ignore_index.

    Returns the number of positions that were masked."""
    N = labels.shape[0]
    k = int(round(frac * N))
    if k == 0:
        return 0
    g = _gen(seed, "cpu")
    pos = torch.randperm(N, generator=g)[:k].to(labels.device)
    labels[pos] = ignore_index
    return k


def packed_document_labels(B: int, T: int, V: int, n_docs: int, pad_tail: int, seed: int,
                           device="cpu", ignore_index=IGNORE_INDEX) -> torch.Tensor:
    """Zipf(1.1) labels for B packed rows of T tokens.

    Each row ends in a padding tail of ``pad_tail`` tokens; the other tokens are
    split into ``n_docs`` documents at seeded cut points.  The padding tail and
    the last token of every document are set to ``ignore_index`` (the token
    after a document's end belongs to the next document, so it has no label)."""
    labels = zipf_labels(B * T, V, 1.1, seed, "cpu").view(B, T)
    g = _gen(seed + 7919, "cpu")
    body = T - pad_tail
    for r in range(B):
        cuts = torch.randperm(body - 2, generator=g)[: n_docs - 1] + 1
        ends = sorted(int(c) for c in cuts) + [body]
        for e in ends:
            labels[r, e - 1] = ignore_index
        labels[r, body:] = ignore_index
    return labels.reshape(-1).to(device)


# --------------------------------------------------------------------------- workloads

def tiny_flce(reduction: str = "sum", device="cpu", seed: int = 1) -> FLCEInputs:
    N, D, V = 256, 128, 1000
    H = normal((N, D), 1.0, torch.float32, seed * 100 + 1, device)
    W = normal((V, D), 0.02, torch.float32, seed * 100 + 2, device)
    labels = uniform_labels(N, V, seed * 100 + 3, device)
    mask_fraction(labels, 0.10, seed * 100 + 4)
    return FLCEInputs("tiny_flce N=256 D=128 V=1000 fp32", H, W, None, labels,
                      IGNORE_INDEX, reduction, None)


def ce_logits_large(device="cpu", seed: int = 2, N: int = 16384, V: int = 128256) -> CEInputs:
    logits = normal((N, V), 2.0, torch.bfloat16, seed * 100 + 1, device)
    labels = uniform_labels(N, V, seed * 100 + 3, device)
    mask_fraction(labels, 0.05, seed * 100 + 4)
    return CEInputs(f"ce_logits N={N} V={V} bf16", logits, labels, IGNORE_INDEX, "sum",
                    None, True)


def small_flce(device="cpu", seed: int = 3) -> FLCEInputs:
    N, D, V = 2 * 1024, 768, 32777
    H = normal((N, D), 1.0, torch.bfloat16, seed * 100 + 1, device)
    W = normal((V, D), 0.02, torch.bfloat16, seed * 100 + 2, device)
    bias = normal((V,), 0.01, torch.bfloat16, seed * 100 + 5, device)
    labels = uniform_labels(N, V, seed * 100 + 3, device)
    return FLCEInputs("small_flce N=2048 D=768 V=32777 bf16 +bias", H, W, bias, labels,
                      IGNORE_INDEX, "mean", None)


def llama3_8b_flce(device="cpu", seed: int = 4, N: int = 8192) -> FLCEInputs:
    D, V = 4096, 128256
    H = normal((N, D), 1.0, torch.bfloat16, seed * 100 + 1, device)
    W = normal((V, D), 0.02, torch.bfloat16, seed * 100 + 2, device)
    labels = zipf_labels(N, V, 1.1, seed * 100 + 3, device)
    masked = mask_fraction(labels, 0.03, seed * 100 + 4)
    return FLCEInputs(f"llama3_8b_flce N={N} D=4096 V=128256 bf16", H, W, None, labels,
                      IGNORE_INDEX, "sum", N - masked)


def long_packed_flce(device="cpu", seed: int = 5, B: int = 4, T: int = 16384) -> FLCEInputs:
    D, V = 5120, 151936
    N = B * T
    H = normal((N, D), 1.0, torch.bfloat16, seed * 100 + 1, device)
    W = normal((V, D), 0.015, torch.bfloat16, seed * 100 + 2, device)
    pad = int(round(1307 * T / 16384))
    labels = packed_document_labels(B, T, V, 4, pad, seed * 100 + 3, device)
    return FLCEInputs(f"long_packed_flce N={N} D=5120 V=151936 bf16", H, W, None, labels,
                      IGNORE_INDEX, "sum", None)


def random_flce(N: int, D: int, V: int, dtype=torch.bfloat16, bias=False, seed: int = 0,
                ignore_frac: float = 0.1, reduction="sum", num_label_tokens=None,
                w_std: float = 0.02, device="cpu") -> FLCEInputs:
    """Free-size FLCE inputs for parity tests (same recipe as the workloads above)."""
    H = normal((N, D), 1.0, dtype, seed * 100 + 1, device)
    W = normal((V, D), w_std, dtype, seed * 100 + 2, device)
    b = normal((V,), 0.01, dtype, seed * 100 + 5, device) if bias else None
    labels = uniform_labels(N, V, seed * 100 + 3, device)
    mask_fraction(labels, ignore_frac, seed * 100 + 4)
    return FLCEInputs(f"random_flce N={N} D={D} V={V}", H, W, b, labels, IGNORE_INDEX,
                      reduction, num_label_tokens)


def random_ce(N: int, V: int, dtype=torch.bfloat16, std: float = 2.0, seed: int = 0,
              ignore_frac: float = 0.05, reduction="sum", num_label_tokens=None,
              inplace_grad=False, ld: Optional[int] = None, device="cpu") -> CEInputs:
    """Free-size given-logits inputs.  With ``ld > V`` the logits are a column
    slice of a wider [N, ld] buffer (row stride ld)."""
    width = V if ld is None else ld
    full = normal((N, width), std, dtype, seed * 100 + 1, device)
    logits = full[:, :V]
    labels = uniform_labels(N, V, seed * 100 + 3, device)
    mask_fraction(labels, ignore_frac, seed * 100 + 4)
    return CEInputs(f"random_ce N={N} V={V}", logits, labels, IGNORE_INDEX, reduction,
                    num_label_tokens, inplace_grad)


WORKLOADS = {
    "tiny_flce": tiny_flce,
    "ce_logits_large": ce_logits_large,
    "small_flce": small_flce,
    "llama3_8b_flce": llama3_8b_flce,
    "long_packed_flce": long_packed_flce,
}


def bf16_bytes_to_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array (host)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def fraction_ignored(labels: torch.Tensor, ignore_index=IGNORE_INDEX) -> float:
    return float((labels == ignore_index).sum().item()) / max(1, labels.numel())

