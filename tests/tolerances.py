"""Parity tolerances of the GPU tests and where each comes from.

Stated by the hot-path specification for bf16 inputs (kept as they are):

* loss: |gpu - ref| <= 1e-3 |ref|;
* grad_H, grad_W, grad_b, dlogits: max relative <= 2e-2 and normwise <= 5e-3
  (dlogits is rounded to the input dtype before the two gradient
  contractions, as Liger-Kernel issue #533's feature pitch casts the chunk's
  gradient to the input dtype);
* n_valid and the label index: exact.

Derived here, tighter, so that a lost piece of the vocabulary fails:

* Per-row lse of the fused linear path, bf16 inputs.  The products of two bf16
  values are exact in fp32, so the logits differ from the fp64 oracle's only by
  the fp32 accumulation over K = D terms (in blocks of 16 inside one MMA), and
  lse is 1-Lipschitz in the max norm of the logits: |d lse| <= max_j |d z_j|
  plus the rounding of the fp32 log-sum-exp itself (a few ulp of |lse|).  Over
  K/16 <= 512 block additions with truncating accumulation the bias is at most
  (K/16) * 2^-24 * max |partial sum|, about 3e-5 at K = 8192 and |z| ~ 1;
  measured at N=8192 D=4096 V=128256 the error is 7.8e-6 (mean 6.5e-6, the
  bias) and 1e-6 or less at D <= 1024.  The bound 2e-5 (1 + |lse|) (2.7e-4 at
  lse ~ 12.6) leaves 17x room, while dropping any one 256-column tile of the
  Llama3-8B vocabulary moves lse by about 1/501 ~ 2e-3, 7x over the bound
  (``tests/test_tolerances.py`` checks this on the oracle).
* Per-row lse of the fused linear path, fp32 inputs (tf32 tensor cores).  The
  tensor core reads the top 19 bits of each fp32 operand (sign, exponent, 10
  explicit mantissa bits): the low 13 bits are dropped, a truncation.  Cut
  operands multiply exactly in fp32 (11 x 11 significand bits), so the kernel
  computes the logits of the cut problem with the bf16 case's accumulation
  error.  The bound is therefore the effect of the cut, evaluated in fp64 on
  the cut operands, plus the bf16 bound:
  |lse_ref(cut H, cut W) - lse_ref(H, W)| + 2e-5 (1 + |lse|).  (Measured on the
  tiny fp32 workload: the GPU's error, max 5.888e-5 and mean 3.609e-5, equals
  the fp64 effect of the truncation, 5.879e-5 and 3.600e-5, to three digits;
  rounding the operands instead would give 8.2e-6.)  Without knowing the
  rounding mode the worst case is 2^-9 max_j sum_k |h_ik| |w_jk| per row
  (each product off by at most 2 * 2^-10 relative), about 5e-3 here:
  ``flce_lse_bound_tf32_worst_case``.
* Per-row loss of the fused linear path: loss_i = lse_i - z_{i,y_i}; both
  terms carry the error above, so the bound is twice the lse bound (for fp32
  inputs twice the worst case, since the cut moves z_y and lse differently).
* Per-row lse of CE on given logits: the logits are exact, only the fp32
  sum of up to 1.5e5 exponentials and the fp32 log remain: 5e-5 (1 + |lse|).
"""
import numpy as np

LOSS_REL = 1e-3
GRAD_MAX_REL = 2e-2
GRAD_NORMWISE = 5e-3
FLCE_LSE_BF16 = 2e-5
CE_LSE = 5e-5
TF32_PRODUCT_REL = 2.0 ** -9


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def flce_lse_bound_bf16(ref_lse):
    """Per-row bound on |lse_gpu - lse_ref| for bf16 inputs."""
    return FLCE_LSE_BF16 * (1.0 + np.abs(np.asarray(ref_lse, dtype=np.float64)))


def tf32_cut(x):
    """fp32 values with the low 13 mantissa bits dropped (as fp64): the
    operand a tf32 tensor core reads."""
    b = np.ascontiguousarray(_f64(x).astype(np.float32)).view(np.uint32)
    return (b & np.uint32(0xFFFFE000)).view(np.float32).astype(np.float64)


def flce_lse_bound_tf32(ref_lse, H, W, bias=None, rows=None):
    """Per-row bound on |lse_gpu - lse_ref| for fp32 inputs on tf32 tensor
    cores: the fp64 effect of cutting H and W to tf32, plus the bf16 bound."""
    import oracle
    Hc = tf32_cut(H if rows is None else H[rows])
    Z = Hc @ tf32_cut(W).T
    if bias is not None:
        Z += _f64(bias)[None, :]
    cut = oracle.logsumexp_rows(Z)
    return np.abs(cut - np.asarray(ref_lse, dtype=np.float64)) + flce_lse_bound_bf16(ref_lse)


def flce_lse_bound_tf32_worst_case(ref_lse, H, W, rows=None):
    """2^-9 max_j sum_k |h_ik| |w_jk| + the bf16 bound: holds for any cut to
    10 explicit mantissa bits (truncation or rounding)."""
    Ha = np.abs(_f64(H if rows is None else H[rows]))
    absprod = (Ha @ np.abs(_f64(W)).T).max(axis=1)
    return TF32_PRODUCT_REL * absprod + flce_lse_bound_bf16(ref_lse)


def flce_lse_bound(ref_lse, H, W, bias=None, rows=None):
    """The bound for the dtype of H (bf16 or fp32)."""
    import torch
    if getattr(H, "dtype", None) == torch.float32:
        return flce_lse_bound_tf32(ref_lse, H, W, bias, rows)
    return flce_lse_bound_bf16(ref_lse)


def check_flce_lse(got_lse, ref_lse, H, W, bias=None, rows=None, what="lse"):
    got = _f64(got_lse)
    ref = np.asarray(ref_lse, dtype=np.float64)
    bound = flce_lse_bound(ref, H, W, bias, rows)
    err = np.abs(got - ref)
    worst = int(np.argmax(err - bound)) if err.size else 0
    assert np.all(err <= bound), (what, float(err[worst]), float(bound[worst]), worst)


def check_flce_loss_rows(got_rows, ref_rows, ref_lse, H, W, rows=None):
    """loss_i = lse_i - z_{i,y_i}: twice the per-row bound on the logits (the
    worst case for fp32 inputs, where the cut moves z_y and lse differently)."""
    import torch
    got = _f64(got_rows)
    ref = np.asarray(ref_rows, dtype=np.float64)
    if getattr(H, "dtype", None) == torch.float32:
        bound = 2.0 * flce_lse_bound_tf32_worst_case(np.asarray(ref_lse), H, W, rows)
    else:
        bound = 2.0 * flce_lse_bound_bf16(np.asarray(ref_lse))
    err = np.abs(got - ref)
    worst = int(np.argmax(err - bound)) if err.size else 0
    assert np.all(err <= bound), ("loss_rows", float(err[worst]), float(bound[worst]), worst)


def check_loss(got, ref, slack=0.0):
    assert abs(got - ref) <= LOSS_REL * abs(ref) + slack, (got, ref)


def check_grad(got, want, name, oracle):
    mr = oracle.max_rel_err(_f64(got), want)
    nw = oracle.normwise_err(_f64(got), want)
    assert mr <= GRAD_MAX_REL and nw <= GRAD_NORMWISE, (name, mr, nw)
