"""The raw tcgen05 contraction against its plain definition (fp64 numpy A @ B.T).

Every operand layout (K-major / MN-major for A and B) in bf16 and fp32 (tf32
tensor cores), with tails in M, N and K, overwrite and accumulate.
Tolerance: each product of two bf16 values is exact in fp32; the error is the
fp32 accumulation over K terms, far below 1e-3 relative.  tf32 rounds each
input to 10 mantissa bits (relative 2^-11 per input), so a K-term dot product
of N(0,1) values has a relative error of about 2^-10 / sqrt(K) of its scale:
2e-3 of max|C| is a safe bound.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lh():
    import lm_head_linear_fwd_gb300 as m
    return m


@pytest.fixture(params=[31, 0], ids=["pair", "single"])
def variant(request, lh):
    """bf16 contractions on CTA pairs (cta_group::2) or on single CTAs."""
    from lm_head_linear_fwd_gb300 import _abi
    prev = _abi.flce_gemm_set_pair(request.param)
    yield request.param
    _abi.flce_gemm_set_pair(prev)


def _ref(A, B, a_mn, b_mn):
    A64 = A.double().cpu().numpy()
    B64 = B.double().cpu().numpy()
    if a_mn:
        A64 = A64.T
    if b_mn:
        B64 = B64.T
    return A64 @ B64.T


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, False), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 520, 200), (1000, 264, 1032),
                                   (2048, 4096, 512)])
def test_gemm_layouts(lh, variant, dtype, a_mn, b_mn, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn((K, M) if a_mn else (M, K), generator=g, device="cuda").to(dtype)
    B = torch.randn((K, N) if b_mn else (N, K), generator=g, device="cuda").to(dtype)
    C = torch.full((M, N), float("nan"), device="cuda")
    st = lh.new_status("cuda")
    if dtype == torch.float32 and (a_mn or b_mn):
        # the tf32 tensor-core path reads K-major operands only
        with pytest.raises(lh.FlceError) as e:
            lh.flce_gemm(A, B, C, a_mn, b_mn, accumulate=False, status=st)
        assert e.value.code == -8
        return
    lh.flce_gemm(A, B, C, a_mn, b_mn, accumulate=False, status=st)
    torch.cuda.synchronize()
    lh.check_status(st)
    ref = _ref(A, B, a_mn, b_mn)
    tol = 1e-4 if dtype == torch.bfloat16 else 2e-3
    err = np.max(np.abs(C.double().cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err < tol, err
    # accumulate: C += A B^T again
    lh.flce_gemm(A, B, C, a_mn, b_mn, accumulate=True, status=st)
    torch.cuda.synchronize()
    err2 = np.max(np.abs(C.double().cpu().numpy() - 2 * ref)) / np.max(np.abs(2 * ref))
    assert err2 < tol, err2


def test_gemm_is_deterministic(lh, variant):
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn(777, 512, generator=g, device="cuda").bfloat16()
    B = torch.randn(900, 512, generator=g, device="cuda").bfloat16()
    C1 = torch.empty(777, 900, device="cuda")
    C2 = torch.empty(777, 900, device="cuda")
    lh.flce_gemm(A, B, C1)
    lh.flce_gemm(A, B, C2)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
