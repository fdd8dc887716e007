"""The derived parity tolerances (tests/tolerances.py) can fail, and hold for
the arithmetic they are derived from.

* A lost 256-column vocabulary tile (one skipped tile of the forward's
  (m, s) merge, or a last partial tile left out) must move some row's lse by
  more than the bound, for every tile, at the vocabulary sizes and logit
  scales of the workloads (the Llama3-8B head: z ~ N(0, (0.02 sqrt 4096)^2),
  V = 128256; the long packed head: z ~ N(0, (0.015 sqrt 5120)^2), V = 151936).
* The tf32 bound holds for products of operands cut to 10 explicit mantissa
  bits (by truncation and by rounding), evaluated in fp64, on the tiny fp32
  workload's inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import tolerances as tol
import workloads as wl

TILE = 256


def _lse_without_each_tile(Z):
    """[n_tiles, N] lse of Z with one 256-column tile left out, from per-tile
    sums (fp64, plain definition)."""
    m = Z.max(axis=1, keepdims=True)
    E = np.exp(Z - m)
    V = Z.shape[1]
    starts = np.arange(0, V, TILE)
    tile_sums = np.add.reduceat(E, starts, axis=1)          # [N, n_tiles]
    total = tile_sums.sum(axis=1, keepdims=True)
    return (m + np.log(total - tile_sums)).T                 # [n_tiles, N]


@pytest.mark.parametrize("V,sigma", [(128256, 0.02 * 4096 ** 0.5), (151936, 0.015 * 5120 ** 0.5),
                                     (131149, 0.02 * 1024 ** 0.5), (40000, 0.02 * 256 ** 0.5)])
def test_a_dropped_vocab_tile_exceeds_the_bf16_lse_bound(V, sigma):
    rng = np.random.default_rng(V)
    Z = rng.standard_normal((8, V)) * sigma
    y = rng.integers(0, V, 8)
    ref = oracle.ce_forward(Z, y)["lse"]
    bound = tol.flce_lse_bound_bf16(ref)
    shifted = _lse_without_each_tile(Z)
    excess = np.abs(shifted - ref[None, :]) / bound[None, :]
    # every tile, left out, moves at least one row's lse past the bound
    assert np.all(excess.max(axis=1) > 1.0), excess.max(axis=1).min()
    # and by a clear margin for the typical tile
    assert np.median(excess.max(axis=1)) > 3.0


def test_half_a_tile_still_exceeds_the_bound_at_the_llama3_vocabulary():
    V, sigma = 128256, 0.02 * 4096 ** 0.5
    rng = np.random.default_rng(3)
    Z = rng.standard_normal((8, V)) * sigma
    ref = oracle.ce_forward(Z, rng.integers(0, V, 8))["lse"]
    # the last 128 columns (half of the last tile) dropped
    cut = oracle.ce_forward(Z[:, :V - 128], np.zeros(8, dtype=np.int64))["lse"]
    assert np.max(np.abs(cut - ref) / tol.flce_lse_bound_bf16(ref)) > 1.0


def _tf32_round(x):
    """fp32 values rounded (half up in magnitude) to 10 explicit mantissa bits."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64) + 0x1000
    return (b & ~np.uint64(0x1FFF)).astype(np.uint32).view(np.float32).astype(np.float64)


def test_tf32_cut_drops_the_low_13_bits():
    x = np.array([1.0 + 2.0 ** -10 + 2.0 ** -11 + 2.0 ** -20, -3.0 - 2.0 ** -9 - 2.0 ** -15,
                  2.0 ** -126 * 1.5], dtype=np.float32)
    np.testing.assert_array_equal(tol.tf32_cut(x), [1.0 + 2.0 ** -10, -3.0 - 2.0 ** -9,
                                                    2.0 ** -126 * 1.5])


@pytest.mark.parametrize("cut", ["truncate", "round"])
def test_tf32_bounds_hold_for_tf32_operands(cut):
    p = wl.tiny_flce("sum")
    ref = oracle.flce_forward(p.H, p.W, None, p.labels)["lse"]
    if cut == "truncate":
        Z = tol.tf32_cut(p.H) @ tol.tf32_cut(p.W).T
    else:
        Z = _tf32_round(p.H.numpy()) @ _tf32_round(p.W.numpy()).T
    emulated = oracle.ce_forward(Z, p.labels)["lse"]
    err = np.abs(emulated - ref)
    worst = tol.flce_lse_bound_tf32_worst_case(ref, p.H, p.W)
    assert np.all(err <= worst)
    if cut == "truncate":
        assert np.all(err <= tol.flce_lse_bound_tf32(ref, p.H, p.W))
    # neither bound is vacuous: both are below a dropped tile of the 1000-word vocabulary
    shifted = _lse_without_each_tile(oracle.flce_logits(p.H, p.W, None, np.arange(p.N)))
    assert np.all(np.abs(shifted - ref[None, :]).max(axis=1) > worst.max())
