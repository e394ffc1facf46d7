"""attn_deviation_noalloc: the deviation measures without a caller workspace.

Some callers cannot allocate device memory for a workspace: a plain C host
program that has no device allocator of its own, or a process whose device
memory is already reserved up front by another framework's caching pool.
For them the library keeps one fixed scratch array on each GPU it is loaded
on.  These checks call the entry point through the C ABI twice in a row and
compare each result with the workspace-based attn_deviation on the same
inputs, within the tolerance the other deviation tests use.  This file is
collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


def _noalloc(eta, a, b):
    res = eta.DevT()
    rc = eta.lib.attn_deviation_noalloc(ctypes.c_void_p(a.data_ptr()), eta._DTYPE[a.dtype],
                                        ctypes.c_void_p(b.data_ptr()), eta._DTYPE[b.dtype], a.numel(),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                        ctypes.byref(res))
    return rc, res


def _same(eta, got, ref):
    for key in ("max_abs", "w1", "mean_abs", "std_abs", "mean_signed"):
        x, y = getattr(got, key), ref[key]
        assert math.isclose(x, y, rel_tol=1e-10, abs_tol=1e-14), (key, x, y)
    assert got.n == ref["n"]


def test_noalloc_matches_workspace_version_twice(eta):
    g = torch.Generator().manual_seed(123)
    # first call: a large input; second call: a smaller one with other dtypes,
    # so that stale contents of the shared scratch from the first call would show
    a1 = torch.randn(1_000_003, generator=g, dtype=torch.float64).cuda()
    b1 = (a1 + 1e-3 * torch.randn(1_000_003, generator=g, dtype=torch.float64).cuda())
    a2 = torch.randn(70_001, generator=g).to(torch.bfloat16).cuda()
    b2 = torch.randn(70_001, generator=g).cuda()
    for a, b in ((a1, b1), (a2, b2)):
        rc, got = _noalloc(eta, a, b)
        assert rc == eta.ATTN_OK
        torch.cuda.synchronize()
        _same(eta, got, eta.attn_deviation(a, b))


def test_noalloc_rejects_sizes_beyond_its_scratch(eta):
    n = eta.DEVIATION_NOALLOC_MAX_N + 1
    a = torch.zeros(n, dtype=torch.float32, device="cuda")
    rc, _ = _noalloc(eta, a, a)
    assert rc == eta.ATTN_ERR_UNSUPPORTED
    rc, got = _noalloc(eta, a[: n - 1], a[: n - 1])   # exactly the limit is accepted
    assert rc == eta.ATTN_OK and got.max_abs == 0.0 and got.w1 == 0.0
