"""Pins for the FP64 oracle, against facts fixed by the pages and by mathematics.

None of these compares the oracle with itself or with the CUDA path.  Each
check is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong sign, a transposed or swapped operand, an off-by-one causal mask, an
ignored mask, a missing rescale) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle



def _embed_row_problem(scores, values):
    """Embed one row of scores s_j and vectors v_j as a causal attention
    problem with d = dv: q_i = e0, k_j = s_j * e0, scale 1.  Row i then sees
    the prefix of length i+1 (top-left causal alignment)."""
    s = np.asarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    n, dv = vals.shape
    d = max(dv, 1)
    q = np.zeros((n, d)); q[:, 0] = 1.0
    k = np.zeros((n, d)); k[:, 0] = s
    v = np.zeros((n, d)); v[:, :dv] = vals
    return q, k, v


@pytest.fixture(scope="module")
def worked(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        return json.load(f)


# --- the tutorial's worked example (yadro-code.ru FlashAttention tutorial) ---

def test_worked_example_blocked_equals_direct(worked):
    """Every causal prefix x every block width: the online merge equals the
    direct stable softmax-weighted sum within 1e-12 (the tutorial's asserts)."""
    scores, values = worked["scores"], worked["values"]
    q, k, v = _embed_row_problem(scores, values)
    O, L = oracle.attn(q, k, v, causal=True, scale=1.0)
    tol = worked["tolerance"]
    for p in worked["prefix_lengths"]:
        direct = O[p - 1, :2]
        for w in worked["widths"]:
            blocked, lse = oracle.blocked_row(scores[:p], values[:p], w)
            for a, b in zip(blocked, direct):
                assert math.isclose(a, b, rel_tol=tol["rel"], abs_tol=tol["abs"]), (p, w, a, b)
            assert math.isclose(lse, L[p - 1], rel_tol=1e-15, abs_tol=1e-12)


def test_worked_example_closed_forms(worked):
    """Hand-derived closed forms for the first two prefixes.
    One visible position: the output is that position's vector and the
    log-sum-exp is its score.  Two positions, scores 1000 and 1001: the
    weights are 1/(1+e) and e/(1+e), so the output is
    [2/(1+e), (3e-1)/(1+e)] and LSE = 1001 + log(1 + 1/e)."""
    q, k, v = _embed_row_problem(worked["scores"], worked["values"])
    O, L = oracle.attn(q, k, v, causal=True, scale=1.0)
    assert O[0, 0] == 2.0 and O[0, 1] == -1.0 and L[0] == 1000.0
    e = math.e
    assert math.isclose(O[1, 0], 2 / (1 + e), rel_tol=1e-13)
    assert math.isclose(O[1, 1], (3 * e - 1) / (1 + e), rel_tol=1e-13)
    assert math.isclose(L[1], 1001 + math.log1p(1 / e), rel_tol=1e-15)
    # the largest score is 1004: naive exp(1004) overflows binary64, the oracle must not
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert 1004.0 < L[4] < 1004.0 + math.log(5.0)


def test_wrong_per_block_average(worked):
    """Averaging independent per-block softmax outputs gives every block the
    same weight: exactly 0.5 on the tutorial's [0,0 | 100,100] case, while the
    whole-row answer is above 0.999."""
    c = worked["wrong_average_case"]
    s = np.array(c["scores"]); vals = np.array(c["values"])
    per_block = []
    for blk in c["blocks"]:
        q, k, v = _embed_row_problem(s[blk], vals[blk])
        O, _ = oracle.attn(q, k, v, causal=False, scale=1.0)
        per_block.append(O[0, 0])
    wrong = (per_block[0] + per_block[1]) / 2
    assert wrong == c["wrong_per_block_average_equals"]
    q, k, v = _embed_row_problem(s, vals)
    O, _ = oracle.attn(q, k, v, causal=False, scale=1.0)
    assert O[0, 0] > c["whole_row_greater_than"]
    # and the online merge with width 2 gets the whole-row answer
    blocked, _ = oracle.blocked_row(s, vals, 2)
    assert math.isclose(blocked[0], O[0, 0], rel_tol=1e-15)


def test_no_rescale_variant_fails():
    """The tutorial's exercise: drop the exp(m - M) rescale and the merge must
    break.  The shortest failing input has two positions with different
    scores and different values: [0, 1] with values [0, 1], one per block,
    merges to 0.5 instead of e/(1+e)."""
    good, _ = oracle.blocked_row([0.0, 1.0], [[0.0], [1.0]], 1)
    bad, _ = oracle.blocked_row([0.0, 1.0], [[0.0], [1.0]], 1, no_rescale=True)
    assert math.isclose(good[0], math.e / (1 + math.e), rel_tol=1e-15)
    assert bad[0] == 0.5
    # one position can never fail: there is nothing to rescale
    one, _ = oracle.blocked_row([3.0], [[7.0]], 1, no_rescale=True)
    assert one[0] == 7.0


def test_no_rescale_breaks_worked_example(worked):
    scores, values = worked["scores"], worked["values"]
    direct, _ = oracle.blocked_row(scores, values, 8)
    bad, _ = oracle.blocked_row(scores, values, 1, no_rescale=True)
    assert np.max(np.abs(bad - direct)) > 0.1


@pytest.mark.parametrize("width", [1, 2, 3, 5, 8])
def test_block_permutation_invariance(width):
    """Merging the blocks in any order gives the same result (the tutorial's
    exercise: permute the blocks, the answer must hold within tolerance)."""
    rng = np.random.default_rng(width)
    n = 37
    s = rng.normal(size=n) * 20
    vals = rng.normal(size=(n, 3))
    ref, lse = oracle.blocked_row(s, vals, width)
    nb = (n + width - 1) // width
    for t in range(5):
        order = rng.permutation(nb)
        out, lse2 = oracle.blocked_row(s, vals, width, block_order=order)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        assert math.isclose(lse2, lse, rel_tol=1e-14)


# --- closed forms and invariants of the definition ---

def test_equal_scores_give_mean_of_v():
    """Q = 0 makes every score equal: the output is the plain mean of the
    visible V rows and the LSE is log(number of visible keys)."""
    rng = np.random.default_rng(1)
    N, d = 9, 4
    q = np.zeros((2, N, d)); k = rng.normal(size=(2, N, d)); v = rng.normal(size=(2, N, d))
    O, L = oracle.attn(q, k, v, causal=False, scale=0.5)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(L, np.log(N), rtol=0, atol=1e-14)
    O, L = oracle.attn(q, k, v, causal=True, scale=0.5)
    for i in range(N):
        np.testing.assert_allclose(O[:, i], v[:, : i + 1].mean(axis=1), rtol=0, atol=1e-14)
        np.testing.assert_allclose(L[:, i], math.log(i + 1), rtol=0, atol=1e-14)


def test_causal_row0_is_v0():
    """Under the causal mask the first query sees only key 0: O = V[0] and
    LSE = scale * <q_0, k_0>."""
    rng = np.random.default_rng(2)
    q, k, v = (rng.normal(size=(3, 11, 8)) for _ in range(3))
    O, L = oracle.attn(q, k, v, causal=True, scale=0.3)
    np.testing.assert_array_equal(O[:, 0], v[:, 0])
    np.testing.assert_allclose(L[:, 0], 0.3 * np.einsum("bd,bd->b", q[:, 0], k[:, 0]), rtol=1e-13, atol=1e-15)


def test_attention_rows_sum_to_one():
    """With V all ones every output element is the row's weight sum, which is 1."""
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(4, 33, 16)) * 3, rng.normal(size=(4, 33, 16)) * 3
    v = np.ones((4, 33, 16))
    mask = np.where(rng.random((4, 33)) < 0.2, -np.inf, rng.normal(size=(4, 33)))
    mask[:, 0] = 0.0
    for causal in (False, True):
        O, _ = oracle.attn(q, k, v, causal=causal, scale=0.25, key_mask=mask)
        np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


def test_fully_masked_rows_are_zero():
    """A row with no allowed key outputs 0 with LSE = -inf and no NaN
    (the definition this library adopts; the tutorial leaves it open)."""
    rng = np.random.default_rng(4)
    q, k, v = (rng.normal(size=(2, 7, 4)) for _ in range(3))
    mask = np.zeros((2, 7)); mask[1, :] = -np.inf          # head 1: every key masked
    O, L = oracle.attn(q, k, v, causal=False, scale=1.0, key_mask=mask)
    assert np.all(O[1] == 0.0) and np.all(L[1] == -np.inf)
    assert np.all(np.isfinite(O[0])) and np.all(np.isfinite(L[0]))
    mask = np.zeros((2, 7)); mask[:, :3] = -np.inf         # causal: rows 0..2 see only masked keys
    O, L = oracle.attn(q, k, v, causal=True, scale=1.0, key_mask=mask)
    assert np.all(O[:, :3] == 0.0) and np.all(L[:, :3] == -np.inf)
    assert not np.any(np.isnan(O)) and not np.any(np.isnan(L))
    np.testing.assert_array_equal(O[:, 3], v[:, 3])        # row 3 sees exactly one allowed key


def test_single_key():
    rng = np.random.default_rng(5)
    q, k, v = (rng.normal(size=(3, 1, 6)) for _ in range(3))
    for causal in (False, True):
        O, L = oracle.attn(q, k, v, causal=causal, scale=0.7)
        np.testing.assert_array_equal(O, v)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_scipy_softmax(causal):
    """Against the library routines: scipy.special.softmax of the scaled,
    masked score matrix times V, and scipy.special.logsumexp."""
    rng = np.random.default_rng(6)
    B, H, N, d = 2, 3, 37, 16
    q, k, v = (rng.normal(size=(B, H, N, d)) for _ in range(3))
    mask = np.where(rng.random((B, H, N)) < 0.1, -np.inf, 0.3 * rng.normal(size=(B, H, N)))
    mask[..., 0] = 0.0
    scale = 1 / math.sqrt(d)
    O, L = oracle.attn(q, k, v, causal=causal, scale=scale, key_mask=mask)
    S = np.einsum("bhid,bhjd->bhij", q, k) * scale + mask[:, :, None, :]
    if causal:
        S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
    P = scipy.special.softmax(S, axis=-1)
    np.testing.assert_allclose(O, P @ v, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, scipy.special.logsumexp(S, axis=-1), rtol=1e-13, atol=1e-13)


def test_permutation_equivariance():
    """Non-causal attention is invariant to permuting the key/value rows
    together and equivariant to permuting the query rows."""
    rng = np.random.default_rng(7)
    q, k, v = (rng.normal(size=(1, 29, 8)) for _ in range(3))
    O, L = oracle.attn(q, k, v, causal=False, scale=0.4)
    pk = rng.permutation(29)
    O2, L2 = oracle.attn(q, k[:, pk], v[:, pk], causal=False, scale=0.4)
    np.testing.assert_allclose(O2, O, rtol=1e-13, atol=1e-14)
    pq = rng.permutation(29)
    O3, L3 = oracle.attn(q[:, pq], k, v, causal=False, scale=0.4)
    np.testing.assert_allclose(O3, O[:, pq], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L3, L[:, pq], rtol=1e-14)


def test_shift_invariance_via_mask():
    """Adding the same constant to every score of a row leaves O unchanged
    and shifts LSE by that constant."""
    rng = np.random.default_rng(8)
    q, k, v = (rng.normal(size=(2, 13, 8)) for _ in range(3))
    O, L = oracle.attn(q, k, v, causal=True, scale=0.5)
    c = 1234.5
    O2, L2 = oracle.attn(q, k, v, causal=True, scale=0.5, key_mask=np.full((2, 13), c))
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L2 - c, L, rtol=0, atol=1e-10)


def test_large_logits_stay_finite():
    """Scores in the 1e3..1e4 range (the adversarial workload's scale) must
    not overflow: the max subtraction keeps every exponent <= 0."""
    rng = np.random.default_rng(9)
    q, k, v = (rng.normal(size=(1, 64, 32)) for _ in range(3))
    O, L = oracle.attn(q * 30, k * 30, v, causal=True, scale=1 / math.sqrt(32))
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert np.max(np.abs(L)) > 1e3
    # each output row is a convex combination of V rows
    assert np.all(O <= v.max(axis=1, keepdims=True) + 1e-12)
    assert np.all(O >= v.min(axis=1, keepdims=True) - 1e-12)


def test_row_subset_matches_full():
    rng = np.random.default_rng(10)
    q, k, v = (rng.normal(size=(2, 2, 19, 8)) for _ in range(3))
    O, L = oracle.attn(q, k, v, causal=True, scale=0.3)
    rows = np.array([0, 5, 18, 19, 40, 75])
    Os, Ls = oracle.attn(q, k, v, causal=True, scale=0.3, rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(Ls, L.reshape(-1)[rows])


# --- deviation measures ---

def _w1_cdf_integral(a, b):
    """W1 as the integral of |F_a(x) - F_b(x)| over x, by brute force on the
    merged support (a different formula from the sorted-pairs one)."""
    pts = np.sort(np.concatenate([a, b]))
    tot = 0.0
    for x0, x1 in zip(pts[:-1], pts[1:]):
        if x1 == x0:
            continue
        Fa = np.count_nonzero(a <= x0) / a.size
        Fb = np.count_nonzero(b <= x0) / b.size
        tot += abs(Fa - Fb) * (x1 - x0)
    return tot


def test_deviation_against_definitions():
    rng = np.random.default_rng(11)
    for n in (1, 2, 7, 50):
        a = rng.normal(size=n); b = rng.normal(size=n) * 2 + 0.3
        r = oracle.deviation(a, b)
        assert r["max_abs"] == np.max(np.abs(a - b))
        assert math.isclose(r["w1"], _w1_cdf_integral(a, b), rel_tol=1e-12, abs_tol=1e-15)
        assert math.isclose(r["w1"], scipy.stats.wasserstein_distance(a, b), rel_tol=1e-12, abs_tol=1e-15)
        assert math.isclose(r["mean_abs"], np.mean(np.abs(a - b)), rel_tol=1e-13)
        assert math.isclose(r["std_abs"], np.std(np.abs(a - b)), rel_tol=1e-10, abs_tol=1e-15)
        assert math.isclose(r["mean_signed"], np.mean(a - b), rel_tol=1e-12, abs_tol=1e-15)


def test_deviation_shift_and_bound():
    """W1(a, a + c) = |c|; W1 <= mean |a - b| for any pairing; W1 ignores order."""
    rng = np.random.default_rng(12)
    a = rng.normal(size=1000)
    r = oracle.deviation(a, a + 0.25)
    assert math.isclose(r["w1"], 0.25, rel_tol=1e-12)
    b = rng.normal(size=1000)
    r = oracle.deviation(a, b)
    assert r["w1"] <= r["mean_abs"] + 1e-15
    r2 = oracle.deviation(a, rng.permutation(a))
    assert r2["w1"] == 0.0
    assert r2["max_abs"] > 0.0
