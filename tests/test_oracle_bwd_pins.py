"""Pins of the oracle's attention gradients (CPU only).

``oracle.attn_bwd`` writes out the chain rule through the softmax (the
gradients that the backward pass of the yadro-code.ru FlashAttention tutorial
recomputes, and whose closeness its checklist asks for).  It is pinned here
against things it does not compute itself:

- central finite differences of L = sum(O * dO), where O comes from the
  forward oracle ``oracle.attn`` (the definition of attention, "Is Flash
  Attention Stable?" §II-A), for every entry of Q, K and V on tiny inputs:
  causal, non-causal, a key mask and a fully masked row;
- the same check catching the two planted mistakes (the softmax Jacobian's
  rank-one term dropped; the scale left out);
- invariances of attention that fix sums of the gradients: the same vector
  added to every key leaves O unchanged (sum_j dK_j = 0); the same vector
  added to every value shifts each non-empty row of O by it
  (sum_j dV_j = sum of dO over those rows); O depends on Q and K only through
  Q K^T (Q^T dQ = dK^T K);
- closed forms: one key (dV = dO, dQ = dK = 0) and Q = 0 (uniform weights:
  dV_j is the dO of each row that sees key j divided by that row's key count,
  dK = 0).
"""
import math

import numpy as np
import pytest

import oracle


def _rand(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, do, causal, scale, mask):
    o, _ = oracle.attn(q, k, v, causal, scale, key_mask=mask, nthreads=1)
    return float(np.sum(o * do))


def _fd_grads(q, k, v, do, causal, scale, mask, h=1e-5):
    grads = []
    for which in range(3):
        base = [q, k, v]
        g = np.zeros_like(base[which])
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (_loss(*plus, do, causal, scale, mask) - _loss(*minus, do, causal, scale, mask)) / (2 * h)
        grads.append(g)
    return grads


def _tiny_case(seed, masked):
    BH, N, d = 2, 6, 4
    q, k, v, do = (_rand(seed + t, (BH, N, d)) for t in range(4))
    mask = None
    if masked:
        mask = np.zeros((BH, N))
        mask[0, 0] = -np.inf     # with causal: row 0 of head 0 sees no key
        mask[1, 3] = -np.inf
        mask[1, 4] = 0.7         # a finite additive term
    return q, k, v, do, mask


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("masked", [False, True])
def test_gradients_match_finite_differences(causal, masked):
    q, k, v, do, mask = _tiny_case(10 + 2 * causal + masked, masked)
    scale = 0.6
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale, key_mask=mask)
    fq, fk, fv = _fd_grads(q, k, v, do, causal, scale, mask)
    for got, want in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.max(np.abs(got - want)) <= 1e-7 * max(1.0, np.max(np.abs(want)))
    if masked and causal:
        # row 0 of head 0 is fully masked: O there is the constant 0
        assert np.all(dq[0, 0] == 0.0)


@pytest.mark.parametrize("plant", [oracle.ORACLE_BWD_PLANT_NO_CENTER, oracle.ORACLE_BWD_PLANT_NO_SCALE])
def test_planted_mistakes_fail_finite_differences(plant):
    q, k, v, do, mask = _tiny_case(20, False)
    scale = 0.6
    dq, dk, _ = oracle.attn_bwd(q, k, v, do, False, scale, plant=plant)
    fq, fk, _ = _fd_grads(q, k, v, do, False, scale, None)
    err = max(np.max(np.abs(dq - fq)), np.max(np.abs(dk - fk)))
    assert err > 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_invariances_fix_gradient_sums(causal):
    BH, N, d = 3, 200, 16
    q, k, v, do = (_rand(30 + t, (BH, N, d)) for t in range(4))
    mask = np.where(np.random.default_rng(34).random((BH, N)) < 0.1, -np.inf, 0.0)
    mask[0, :2] = -np.inf                     # causal rows 0, 1 of head 0: no visible key
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale, key_mask=mask)
    _, lse = oracle.attn(q, k, v, causal, scale, key_mask=mask)
    visible = np.isfinite(lse)                # rows with at least one allowed key
    for h in range(BH):
        assert np.max(np.abs(dk[h].sum(axis=0))) <= 1e-11 * N
        want_dv = (do[h] * visible[h][:, None]).sum(axis=0)
        assert np.max(np.abs(dv[h].sum(axis=0) - want_dv)) <= 1e-11 * N
        lhs = q[h].T @ dq[h]
        rhs = dk[h].T @ k[h]
        assert np.max(np.abs(lhs - rhs)) <= 1e-10 * N
    assert visible.all() != causal           # causal: the planted empty rows are there


def test_single_key():
    q, k, v, do = (_rand(40 + t, (2, 1, 8)) for t in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, 0.3)
    assert np.array_equal(dv, do)
    assert np.max(np.abs(dq)) <= 1e-15 and np.max(np.abs(dk)) <= 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_weights(causal):
    BH, N, d = 2, 50, 8
    k, v, do = (_rand(50 + t, (BH, N, d)) for t in range(3))
    q = np.zeros((BH, N, d))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.5)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    w = do / counts[None, :, None]            # each row spreads its dO evenly over its keys
    if causal:
        want = np.flip(np.cumsum(np.flip(w, axis=1), axis=1), axis=1)   # keys j see rows i >= j
    else:
        want = np.broadcast_to(w.sum(axis=1, keepdims=True), w.shape)
    assert np.max(np.abs(dv - want)) <= 1e-12
    assert np.max(np.abs(dk)) <= 1e-15
    # dQ_i = scale * sum_j P_ij (G_ij - mean_j G_ij) k_j with uniform P_ij
    i = N - 1
    G = do[0, i] @ v[0].T
    want_dq = 0.5 * ((G - G.mean()) / N) @ k[0]
    assert np.max(np.abs(dq[0, i] - want_dq)) <= 1e-12


def test_head_subset_matches_all_heads():
    q, k, v, do = (_rand(60 + t, (4, 33, 8)) for t in range(4))
    full = oracle.attn_bwd(q, k, v, do, True, 0.4)
    sub = oracle.attn_bwd(q, k, v, do, True, 0.4, heads=[3, 1])
    for a, b in zip(full, sub):
        assert np.array_equal(a[[3, 1]], b)
