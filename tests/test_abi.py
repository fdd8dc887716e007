"""Host-side checks of the C ABI (no GPU needed).

The library loads, exports every function the headers declare, and rejects
bad arguments with the documented status codes before touching the device.
Only argument combinations that fail host validation are passed here, and the
validation tests are skipped on a machine with a GPU so that no call with a
stand-in pointer can ever reach a kernel.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in ("flce.h", "flce_gemm.h")]


def _declared():
    names = []
    for h in HEADERS:
        src = open(h).read()
        names += re.findall(r"FLCE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from lm_head_linear_fwd_gb300 import _abi
    return _abi.load()


def test_headers_declare_the_boundary():
    names = set(_declared())
    for n in ("ce_logits_fwd", "ce_logits_bwd", "ce_logits_workspace_bytes", "flce_fwd",
              "flce_bwd", "flce_workspace_bytes", "flce_default_chunk", "flce_status_string",
              "flce_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    from lm_head_linear_fwd_gb300 import _abi
    assert set(_abi.EXPORTED) == set(_declared())


def test_status_strings(lib):
    from lm_head_linear_fwd_gb300 import _abi
    for code in range(0, -11, -1):
        assert _abi.status_string(code).startswith("FLCE")


def test_workspace_sizes(lib):
    from lm_head_linear_fwd_gb300 import _abi
    assert _abi.ce_logits_workspace_bytes(0, 10) == 0
    assert _abi.ce_logits_workspace_bytes(16384, 128256) >= 16384 * 4
    n = _abi.flce_workspace_bytes(0, 8192, 4096, 128256, 0)
    chunk = _abi.flce_default_chunk(0, 8192, 4096, 128256)
    assert chunk % 128 == 0 and 128 <= chunk <= 8192
    # the workspace holds the dZ chunk buffer (bf16)
    assert n >= chunk * 128256 * 2
    # explicit row chunks and vocabulary slices size their own workspaces: a
    # slice holds the dZ of all rows for its columns and the fp32 grad_H
    assert _abi.flce_workspace_bytes(0, 8192, 4096, 128256, 4096) >= 4096 * 128256 * 2
    assert _abi.flce_workspace_bytes(0, 8192, 4096, 128256, -256) >= 8192 * 256 * 2 + 8192 * 4096 * 4
    # the one-call path always chunks rows: a negative chunk means its default
    assert (_abi.flce_fwd_bwd_workspace_bytes(0, 8192, 4096, 128256, -256) ==
            _abi.flce_fwd_bwd_workspace_bytes(0, 8192, 4096, 128256, 0))
    assert _abi.flce_default_chunk(0, 2048, 768, 32777) == 2048
    assert _abi.flce_default_chunk(7, 8, 8, 8) == 0
    # with the default chunk, the workspaces of the recomputing and of the
    # one-call path stay within one [2048, V] fp32 tile (bf16 inputs), at the
    # shapes of the workloads and at a few others
    for N, D, V in ((8192, 4096, 128256), (65536, 5120, 151936), (2048, 768, 32777),
                    (256, 128, 1000), (100000, 4096, 50257), (4096, 8192, 262144)):
        budget = 2048 * V * 4
        for fn in (_abi.flce_workspace_bytes, _abi.flce_fwd_bwd_workspace_bytes):
            assert fn(0, N, D, V, 0) <= budget, (fn.__name__, N, D, V)
    assert _abi.flce_workspace_bytes(7, 8, 8, 8, 0) == 0  # bad dtype


no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="host-validation tests use stand-in pointers; CPU only")
FAKE = 0x10000  # never dereferenced: every call below fails host validation first


@no_gpu
def test_ce_fwd_rejects_bad_arguments(lib):
    from lm_head_linear_fwd_gb300 import _abi
    args = dict(logits=FAKE, dt=0, N=4, V=10, ld=10, labels=FAKE, ig=-100, red=0, nlt=-1,
                loss=FAKE, nv=FAKE, lse=FAKE, rows=None, zl=None, ws=FAKE, wsb=1024,
                status=FAKE, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return _abi.ce_logits_fwd(*a.values())
    assert call(dt=5) == -3
    assert call(red=7) == -1
    assert call(V=0) == -2
    assert call(ld=9) == -2
    assert call(N=-1) == -2
    assert call(labels=None) == -1
    assert call(status=None) == -1
    assert call(ws=None) == -6
    assert call(wsb=8) == -6
    assert call(logits=FAKE + 1) == -4


@no_gpu
def test_ce_bwd_rejects_bad_arguments(lib):
    from lm_head_linear_fwd_gb300 import _abi
    base = [FAKE, 0, 4, 10, 10, FAKE, -100, 0, -1, FAKE, FAKE, FAKE, 1, FAKE, 10, FAKE, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return _abi.ce_logits_bwd(*a)
    assert call(12, 2) == -1            # inplace flag not 0/1
    assert call(13, FAKE + 4096) == -1  # in place but grad pointer differs
    assert call(14, 12) == -1           # in place but row strides differ
    assert call(10, None) == -1         # n_valid missing
    assert call(1, 3) == -3
    # lse may be NULL (formed again in the kernel), but not for a vocabulary
    # shard, whose rows need the global lse
    shard = [FAKE, 0, 4, 10, 10, 0, 20, FAKE, -100, 0, -1, None, FAKE, FAKE, 0, FAKE + 4096, 10,
             FAKE, None]
    assert _abi.ce_logits_bwd_shard(*shard) == -1
    shard[11] = FAKE
    shard[6] = 5  # V_total < vocab_offset + V_shard
    assert _abi.ce_logits_bwd_shard(*shard) == -2


@no_gpu
def test_ce_fwd_bwd_rejects_bad_arguments(lib):
    from lm_head_linear_fwd_gb300 import _abi
    G = FAKE + (1 << 20)  # a separate gradient buffer
    args = dict(logits=FAKE, dt=0, N=4, V=10, ld=10, labels=FAKE, ig=-100, red=0, nlt=-1,
                g=None, loss=FAKE, nv=FAKE, lse=None, inplace=0, grad=G, ldg=10, ws=FAKE,
                wsb=1024, status=FAKE, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return _abi.ce_logits_fwd_bwd(*a.values())
    assert call(dt=5) == -3
    assert call(loss=None) == -1
    assert call(status=None) == -1
    assert call(inplace=2) == -1
    assert call(inplace=1) == -1               # in place, but the gradient is elsewhere
    assert call(inplace=1, grad=FAKE, ldg=12) == -1
    assert call(grad=FAKE + 4) == -1           # out of place, overlapping the logits
    assert call(grad=None) == -1
    assert call(ldg=9) == -2
    assert call(ws=None) == -6
    assert call(wsb=8) == -6
    assert call(ws=FAKE + 8) == -4
    assert _abi.ce_logits_fwd_bwd_workspace_bytes(4, 10) >= 2 * 4 * 4
    assert _abi.ce_logits_fwd_bwd_workspace_bytes(0, 10) == 0


@no_gpu
def test_flce_rejects_bad_arguments(lib):
    from lm_head_linear_fwd_gb300 import _abi
    base = [FAKE, FAKE, None, 0, 256, 128, 1000, FAKE, -100, 0, -1, FAKE, FAKE, FAKE, None, None,
            FAKE, 1 << 30, FAKE, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return _abi.flce_fwd(*a)
    assert call(4, -1) == -2         # N < 0 (N = 0, an empty batch, is valid)
    assert call(1, None) == -1       # W missing
    assert call(5, 4) == -2          # D < 8
    assert call(5, 100) == -4        # D*2 not a multiple of 16
    assert call(0, FAKE + 2) == -4   # H not 16-byte aligned
    assert call(3, 9) == -3
    assert call(17, 16) == -6        # workspace too small
    assert call(2, FAKE + 1) == -4   # bias misaligned
    bb = [FAKE, FAKE, None, 0, 256, 128, 1000, FAKE, -100, 0, -1, FAKE, FAKE, FAKE, 100, FAKE,
          FAKE, 0, None, FAKE, 1 << 30, FAKE, None]
    b2 = list(bb)
    b2[14] = 100                     # chunk not a multiple of 128 (and < N)
    assert _abi.flce_bwd(*b2) == -2
    b3 = list(bb)
    b3[17] = 2
    assert _abi.flce_bwd(*b3) == -1
    b4 = list(bb)
    b4[14] = -300                    # vocabulary slice not a multiple of 256
    assert _abi.flce_bwd(*b4) == -2
    b5 = list(bb)
    b5[3], b5[14] = 1, -256          # vocabulary slices with fp32 inputs
    assert _abi.flce_bwd(*b5) == -8


@no_gpu
def test_gemm_rejects_bad_arguments(lib):
    from lm_head_linear_fwd_gb300 import _abi
    base = [0, 0, 0, 64, 64, 64, FAKE, 64, FAKE, 64, FAKE, 64, 0, FAKE, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return _abi.flce_gemm(*a)
    assert call(7, 60) == -4   # lda*2 not a multiple of 16
    assert call(7, 32) == -2   # lda < K
    assert call(1, 3) == -1
    assert call(3, 0) == -2
    assert call(0, 2) == -3


def test_product_path_has_no_fallback():
    """The package never imports the oracle, and a missing library raises."""
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "lm_head_linear_fwd_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f
    code = ("import lm_head_linear_fwd_gb300._abi as a\na._lib = None\n"
            "try:\n    a.load('/nonexistent/libflce.so')\nexcept ImportError:\n    print('raised')\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert "raised" in out.stdout
    ctypes  # noqa: B018  (ctypes import kept for symbol lookups above)


def test_front_ends_check_leading_shapes():
    # shape checks of the autograd front ends happen on the host, before any launch
    import torch
    import lm_head_linear_fwd_gb300 as lh
    x = torch.zeros(2, 3, 10)
    with pytest.raises(ValueError):
        lh.ce_logits(x, torch.zeros(6, dtype=torch.int64))
    with pytest.raises(ValueError):
        lh.ce_logits(torch.zeros(10), torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError):
        lh.flce(x, torch.zeros(10, 10), torch.zeros(2, 3, dtype=torch.int64),
                mask=torch.ones(6))
