"""Block-sparse forward on the GPU (attn_fwd_block_sparse) against the FP64
oracle's block-sparse reading: scores outside the marked 128 x 128
(query block, key block) pairs are -inf before the softmax.

Tolerances are those of the bf16 forward: O max-abs 2e-2, LSE
1e-3 + 2^-8 + 2e-6 |LSE| (the forward's bf16 LSE bound); rows that see no allowed key give O = 0,
LSE = -inf."""
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


def _check(eta, B, H, N, d, causal, bm, seed, key_mask=None, rows=None):
    q, k, v = workloads.make_qkv(B, H, N, d, "bf16", seed)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = eta.attn_fwd_block_sparse(q.cuda(), k.cuda(), v.cuda(), bm.cuda(), causal, scale,
                                       key_mask=key_mask.cuda() if key_mask is not None else None)
    assert eta.attn_status() == 0
    assert eta.attn_last_variant().endswith("bsparse")
    o_ref, l_ref = oracle.attn(q, k, v, causal, scale, key_mask=key_mask, block_mask=bm, rows=rows)
    og = o.double().cpu().numpy().reshape(-1, d)
    lg = lse.double().cpu().numpy().reshape(-1)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    o_ref = o_ref.reshape(-1, d)
    l_ref = l_ref.reshape(-1)
    assert not np.isnan(og).any()
    assert np.max(np.abs(og - o_ref)) <= 2e-2
    inf_ref = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lg), inf_ref)
    assert np.all(og[inf_ref] == 0.0)
    fin = ~inf_ref
    assert np.all(np.abs(lg[fin] - l_ref[fin]) <= 1e-3 + 2.0 ** -8 + 2e-6 * np.abs(l_ref[fin]))
    return inf_ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,density", [(300, 0.5), (1000, 0.3), (1000, 0.8), (2049, 0.4)])
def test_bsparse_random_masks(eta, d, causal, N, density):
    bm = workloads.make_block_mask(1, 3, N, density, seed=N + d)
    _check(eta, 1, 3, N, d, causal, bm, seed=N)


def test_bsparse_all_blocks_equals_dense(eta):
    N = 777
    bm = torch.ones((2, 2, 7, 7), dtype=torch.uint8)
    _check(eta, 2, 2, N, 128, False, bm, seed=1)
    _check(eta, 2, 2, N, 128, True, bm, seed=1)


def test_bsparse_empty_block_rows_and_key_mask(eta):
    B, H, N, d = 1, 4, 1000, 64
    bm = workloads.make_block_mask(B, H, N, 0.5, seed=3)
    bm[0, 1, 2, :] = 0              # head 1, query rows 256..383: no block at all
    bm[0, 2, :, :] = 0              # head 2: nothing
    bm[0, 3, 0, :] = 0              # head 3: the first query tile of a CTA empty, its partner not
    bm[0, 3, 1, 3] = 1
    key_mask = workloads.make_key_mask(B, H, N, 0.1, seed=3)
    inf_ref = _check(eta, B, H, N, d, False, bm, seed=3, key_mask=key_mask)
    rows = inf_ref.reshape(H, N)
    assert rows[1, 256:384].all() and rows[2].all() and rows[3, :128].all()


def test_bsparse_local_window_long(eta):
    """1 x 8 x 8192 x 128, sliding window of +-2 blocks plus a global first
    block; parity on a seeded row sample."""
    B, H, N, d = 1, 8, 8192, 128
    bm = workloads.make_block_mask(B, H, N, pattern="local", window=2)
    rows = workloads.sample_rows(B, H, N, 0.02, seed=5)
    _check(eta, B, H, N, d, False, bm, seed=5, rows=rows)


def test_bsparse_rejects(eta):
    q = torch.zeros((1, 1, 256, 64), dtype=torch.float32, device="cuda")
    bm = torch.ones((1, 1, 2, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(eta.AttnError):
        eta.attn_fwd_block_sparse(q, q, q, bm)                 # float32: bf16 only
    qb = torch.zeros((1, 1, 256, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(eta.AttnError):
        eta.attn_fwd_block_sparse(qb, qb, qb, bm)              # d = 96
    with pytest.raises(ValueError):
        eta.attn_fwd_block_sparse(q.bfloat16(), q.bfloat16(), q.bfloat16(), bm[:, :, :1])   # wrong mask size


@pytest.mark.parametrize("d", [64, 128])
def test_bsparse_finite_key_mask(eta, d):
    """Finite key-mask values (ordinary, tiny, large negative, -inf) on top of
    a random block mask: the mask enters S inside the MMA as in the dense path."""
    B, H, N = 1, 3, 1000
    g = torch.Generator().manual_seed(d)
    key_mask = torch.empty(B, H, N).uniform_(-6.0, 3.0, generator=g)
    sel = torch.rand(B, H, N, generator=g)
    key_mask = torch.where(sel < 0.05, torch.full_like(key_mask, float("-inf")), key_mask)
    key_mask = torch.where((sel >= 0.05) & (sel < 0.10), key_mask - 200.0, key_mask)
    bm = workloads.make_block_mask(B, H, N, 0.5, seed=d + 1)
    _check(eta, B, H, N, d, False, bm, seed=d + 2, key_mask=key_mask)
    _check(eta, B, H, N, d, True, bm, seed=d + 3, key_mask=key_mask)


def test_bsparse_longest_list(eta):
    """N = 131072: 1024 key blocks, the length a unit's key-tile list can
    hold; a sliding window plus block 0, and one query block marking every
    key block (its unit lists all 1024 tiles)."""
    B, H, N, d = 1, 1, 131072, 64
    bm = workloads.make_block_mask(B, H, N, pattern="local", window=1)
    bm[0, 0, 500, :] = 1
    rows = workloads.sample_rows(B, H, N, 32 / N, seed=3, extra=[500 * 128, 500 * 128 + 127, N - 1])
    _check(eta, B, H, N, d, False, bm, seed=5, rows=rows)
