"""Pins of the oracle's block-sparse reading (CPU only).

The yadro-code.ru FlashAttention tutorial notes that the method's paper also
treats a block-sparse extension.  ``oracle.attn(..., block_mask=...)`` reads it
as: the (query block, key block) pairs marked in the mask take part and every
other score is -inf before the softmax.  Pinned against things the oracle's C
code does not compute itself:

- a direct numpy evaluation of softmax over the scores with the block mask
  expanded to an explicit N x N mask (np.kron), on tiny inputs with small
  blocks and a ragged last block;
- a mask marking every block gives exactly the dense result;
- a query block with no marked key block gives O = 0, LSE = -inf (a fully
  masked row);
- the lower block triangle together with the causal rule gives the causal
  result (every key a causal row sees lies in a marked block).
"""
import numpy as np
import pytest

import oracle


def _rand(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _numpy_reference(q, k, v, scale, dense_mask, causal):
    BH, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.full((BH, N), -np.inf)
    for h in range(BH):
        s = scale * q[h] @ k[h].T
        allowed = dense_mask[h].astype(bool)
        if causal:
            allowed &= np.tril(np.ones((N, N), dtype=bool))
        s = np.where(allowed, s, -np.inf)
        for i in range(N):
            if not allowed[i].any():
                continue
            m = s[i].max()
            w = np.exp(s[i] - m)
            o[h, i] = (w @ v[h]) / w.sum()
            lse[h, i] = m + np.log(w.sum())
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_matches_numpy_with_explicit_mask(causal):
    BH, N, d, bq, bk = 3, 50, 8, 8, 6        # 7 x 9 blocks, ragged last block both ways
    q, k, v = (_rand(70 + t, (BH, N, d)) for t in range(3))
    nqb, nkb = -(-N // bq), -(-N // bk)
    bm = (np.random.default_rng(73).random((BH, nqb, nkb)) < 0.5).astype(np.uint8)
    bm[1, 2, :] = 0                           # query rows 16..23 of head 1: no block
    dense = np.stack([np.kron(bm[h], np.ones((bq, bk), dtype=np.uint8))[:N, :N] for h in range(BH)])
    want_o, want_l = _numpy_reference(q, k, v, 0.4, dense, causal)
    got_o, got_l = oracle.attn(q, k, v, causal, 0.4, block_mask=bm, block=(bq, bk))
    assert np.max(np.abs(got_o - want_o)) <= 1e-12
    fin = np.isfinite(want_l)
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.max(np.abs(got_l[fin] - want_l[fin])) <= 1e-12
    assert np.all(got_o[1, 16:24] == 0.0) and np.all(np.isneginf(got_l[1, 16:24]))


def test_all_blocks_marked_is_dense():
    q, k, v = (_rand(80 + t, (2, 300, 16)) for t in range(3))
    bm = np.ones((2, 3, 3), dtype=np.uint8)
    a = oracle.attn(q, k, v, False, 0.25, block_mask=bm)
    b = oracle.attn(q, k, v, False, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_lower_block_triangle_with_causal_is_causal():
    q, k, v = (_rand(90 + t, (2, 300, 16)) for t in range(3))
    bm = np.broadcast_to(np.tril(np.ones((3, 3), dtype=np.uint8)), (2, 3, 3)).copy()
    a = oracle.attn(q, k, v, True, 0.25, block_mask=bm)
    b = oracle.attn(q, k, v, True, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # the upper triangle alone leaves causal rows only their diagonal blocks
    up = np.broadcast_to(np.triu(np.ones((3, 3), dtype=np.uint8)), (2, 3, 3)).copy()
    c = oracle.attn(q, k, v, True, 0.25, block_mask=up)
    dense = np.stack([np.kron(up[h], np.ones((128, 128), dtype=np.uint8))[:300, :300] for h in range(2)])
    want_o, _ = _numpy_reference(q, k, v, 0.25, dense, True)
    assert np.max(np.abs(c[0] - want_o)) <= 1e-12
