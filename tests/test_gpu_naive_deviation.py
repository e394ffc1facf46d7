"""GPU checks of the materialising baseline and the deviation kernels."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


@pytest.mark.parametrize("dtype,tol", [("f32", 1e-5), ("bf16", 2e-2)])
@pytest.mark.parametrize("causal", [False, True])
def test_naive_vs_oracle(eta, dtype, tol, causal):
    B, H, N, d = 2, 3, 333, 64
    q, k, v = workloads.make_qkv(B, H, N, d, dtype, 21)
    mask = workloads.make_key_mask(B, H, N, 0.05, seed=21)
    mask[1, 0, :] = float("-inf")
    dev = torch.device("cuda")
    o, lse = eta.attn_naive_fwd(q.to(dev), k.to(dev), v.to(dev), causal, 1 / math.sqrt(d), mask.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn(q, k, v, causal, 1 / math.sqrt(d), key_mask=mask)
    og = o.double().cpu().numpy()
    assert not np.isnan(og).any()
    assert np.abs(og - o_ref).max() <= tol
    lg = lse.double().cpu().numpy()
    np.testing.assert_array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    assert np.all(og[np.isneginf(lse_ref)] == 0.0)


def _dev_check(eta, a, b):
    r = eta.attn_deviation(a.cuda(), b.cuda())
    ref = oracle.deviation(a, b)
    for key in ("max_abs", "w1", "mean_abs", "std_abs", "mean_signed"):
        x, y = r[key], ref[key]
        if math.isnan(y) or math.isinf(y):
            assert (math.isnan(x) and math.isnan(y)) or x == y, (key, x, y)
            continue
        # float64 sums in a different order: agreement to ~1e-10 relative
        assert math.isclose(x, y, rel_tol=1e-10, abs_tol=1e-14), (key, x, y)
    assert r["n"] == a.numel()


@pytest.mark.parametrize("n", [1, 2, 1000, 4096, 4097, 100_003])
def test_deviation_random(eta, n):
    g = torch.Generator().manual_seed(n)
    a = torch.randn(n, generator=g, dtype=torch.float64)
    b = a + 1e-3 * torch.randn(n, generator=g, dtype=torch.float64)
    _dev_check(eta, a, b)
    _dev_check(eta, a, torch.randn(n, generator=g, dtype=torch.float64) * 3)


def test_deviation_mixed_dtypes_and_adversarial(eta):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(50_000, generator=g)
    a = x.to(torch.bfloat16)
    b = x.to(torch.float32)
    _dev_check(eta, a, b)
    # ties, signed zeros, denormals, equal infinities on both sides
    vals = torch.tensor([0.0, -0.0, 1e-310, -1e-310, 5e-324, float("-inf"), float("inf"), 1.0, 1.0, -1.0],
                        dtype=torch.float64)
    a = vals.repeat(997)
    b = a.flip(0).clone()
    b[::7] = a[::7]
    _dev_check(eta, a, b)
    c = a.clone()
    _dev_check(eta, a, c)  # identical: everything zero


def test_deviation_large_sort(eta):
    """A sort spanning thousands of radix blocks (and all 8 digit passes)."""
    g = torch.Generator().manual_seed(3)
    n = 3_000_017
    a = torch.randn(n, generator=g, dtype=torch.float32) * torch.exp(4 * torch.randn(n, generator=g))
    b = torch.randn(n, generator=g, dtype=torch.float32)
    _dev_check(eta, a, b)
