"""The seeded input generators (CPU only): same seed, same bits; the stated
recipe (N(0,1) float32 draws rounded to the storage dtype, Q and K scaled by
the logit factor); masks with the stated structure."""
import numpy as np
import pytest
import torch

import workloads


def test_qkv_are_reproducible_and_rounded_from_float32_draws():
    a = workloads.make_qkv(1, 2, 50, 16, "bf16", seed=3)
    b = workloads.make_qkv(1, 2, 50, 16, "bf16", seed=3)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.bfloat16 and x.is_contiguous()
    g = torch.Generator(device="cpu").manual_seed(3)
    q32 = torch.randn((1, 2, 50, 16), generator=g, dtype=torch.float32)
    assert torch.equal(a[0], q32.to(torch.bfloat16))
    c = workloads.make_qkv(1, 2, 50, 16, "bf16", seed=4)
    assert not torch.equal(a[0], c[0])


def test_logit_scale_applies_to_q_and_k_only():
    q1, k1, v1 = workloads.make_qkv(1, 1, 40, 8, "f32", seed=5)
    q30, k30, v30 = workloads.make_qkv(1, 1, 40, 8, "f32", seed=5, qk_scale=30.0)
    assert torch.allclose(q30, q1 * 30) and torch.allclose(k30, k1 * 30) and torch.equal(v30, v1)


def test_grad_out_has_its_own_stream():
    do = workloads.make_grad_out(1, 2, 30, 8, "f32", seed=0)
    q, k, v = workloads.make_qkv(1, 2, 30, 8, "f32", seed=0)
    assert not any(torch.equal(do, t) for t in (q, k, v))
    assert torch.equal(do, workloads.make_grad_out(1, 2, 30, 8, "f32", seed=0))


def test_key_mask_structure():
    m = workloads.make_key_mask(1, 8, 1000, 0.05, seed=1)
    assert m.dtype == torch.float32 and m.shape == (1, 8, 1000)
    vals = torch.unique(m)
    assert set(vals.tolist()) <= {0.0, float("-inf")}
    # heads 0 and 4: keys 0..3 always masked (causal rows 0..3 see no key there)
    assert torch.all(torch.isinf(m[0, 0, :4])) and torch.all(torch.isinf(m[0, 4, :4]))
    frac = torch.isinf(m[0, 1:4]).float().mean().item()
    assert 0.02 < frac < 0.08


@pytest.mark.parametrize("N", [128, 300, 1000])
def test_block_mask_patterns(N):
    nb = -(-N // 128)
    r = workloads.make_block_mask(2, 3, N, 0.5, seed=2)
    assert r.dtype == torch.uint8 and r.shape == (2, 3, nb, nb)
    assert torch.equal(r, workloads.make_block_mask(2, 3, N, 0.5, seed=2))
    loc = workloads.make_block_mask(1, 2, N, pattern="local", window=1)
    i = np.arange(nb)
    want = ((np.abs(i[:, None] - i[None, :]) <= 1) | (i[None, :] == 0)).astype(np.uint8)
    assert np.array_equal(loc[0, 0].numpy(), want) and torch.equal(loc[0, 0], loc[0, 1])
