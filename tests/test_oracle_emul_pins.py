"""Pins of the oracle's number-format emulation (CPU only).

The emulation restates the paper's numerical re-implementation ("Is Flash
Attention Stable?" §III, §IV-A Fig. 3): attention with every tensor
operation's result rounded to a chosen format.  It is pinned here against
things it does not compute itself:

- its rounding function against the IEEE conversions numpy and torch perform
  (binary32, binary16, bfloat16), including ties, subnormals and overflow;
- at binary64 both emulated algorithms against the direct FP64 definition of
  attention (``oracle.attn``), for every key-block width;
- the trend the paper reports in Fig. 3: the FlashAttention-vs-baseline
  deviation shrinks as the format's fraction bits grow;
- below binary64, rows worked by hand in a coarse format (2 fraction bits,
  5 exponent bits; ``tests/golden/emul_e5m2_rows.json``), which every
  planted mistake in the oracle's rounding (a left-out, moved or duplicated
  fl()) fails.
"""
import math

import numpy as np
import pytest

import oracle


def _wide_values(rng, n, lo, hi):
    """Random doubles with binary exponents spread over [lo, hi)."""
    e = rng.uniform(lo, hi, n)
    return np.where(rng.random(n) < 0.5, -1.0, 1.0) * np.exp2(e)


def test_round_fp32_matches_ieee_conversion():
    rng = np.random.default_rng(1)
    x = _wide_values(rng, 20000, -160, 130)   # subnormal float32 .. overflow
    with np.errstate(over="ignore"):
        want = x.astype(np.float32).astype(np.float64)
    got = oracle.round_fmt(x, 23, 8)
    assert np.array_equal(got, want)


def test_round_fp32_ties_go_to_even():
    rng = np.random.default_rng(2)
    f = rng.standard_normal(5000).astype(np.float32)
    nxt = np.nextafter(f, np.float32(np.inf))
    mid = (f.astype(np.float64) + nxt.astype(np.float64)) / 2.0   # exact in binary64
    want = mid.astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.round_fmt(mid, 23, 8), want)
    # the even neighbour wins: its last fraction bit is 0
    bits = want.astype(np.float32).view(np.uint32)
    assert np.all(bits & 1 == 0)


def test_round_fp16_matches_ieee_conversion():
    rng = np.random.default_rng(3)
    x = _wide_values(rng, 20000, -28, 18)     # binary16 subnormals .. overflow
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float64)
    got = oracle.round_fmt(x, 10, 5)
    assert np.array_equal(got, want)
    assert oracle.round_fmt(np.array([65519.0, 65520.0]), 10, 5).tolist() == [65504.0, math.inf]


def test_round_bf16_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    x32 = _wide_values(rng, 20000, -140, 127).astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_fmt(x32.astype(np.float64), 7, 8)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "tf32", "fp32"])
def test_round_is_idempotent_odd_and_monotone(fmt):
    mb, eb = oracle.FORMATS[fmt]
    emax = 2 ** (eb - 1) - 1
    rng = np.random.default_rng(5)
    x = np.sort(_wide_values(rng, 4000, max(-20, 1 - emax), min(20, emax)))   # normal range
    y = oracle.round_fmt(x, mb, eb)
    assert np.array_equal(oracle.round_fmt(y, mb, eb), y)
    assert np.array_equal(oracle.round_fmt(-x, mb, eb), -y)
    assert np.all(np.diff(y) >= 0)
    # relative error within half a unit in the last place (normal range)
    rel = np.abs(y - x) / np.abs(x)
    assert rel.max() <= 2.0 ** -(mb + 1) * (1 + 1e-12)


def _case(seed, BH, N, d):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((BH, N, d)) for _ in range(3))
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Bc", [1, 7, 64, 300])
def test_emul_fp64_equals_definition(causal, Bc):
    q, k, v = _case(6, 2, 150, 16)
    scale = 0.25
    want, _ = oracle.attn(q, k, v, causal, scale)
    for algo in (0, 1):
        got = oracle.emul(q, k, v, causal, scale, algo, Bc, 52, 11)
        assert np.max(np.abs(got - want)) <= 1e-12, (algo, Bc)


def test_emul_fp64_masked_and_fully_masked_rows():
    q, k, v = _case(7, 2, 64, 8)
    mask = np.where(np.random.default_rng(8).random((2, 64)) < 0.2, -np.inf, 0.0)
    mask[0, :4] = -np.inf                      # causal rows 0..3 of head 0 see no key
    want, _ = oracle.attn(q, k, v, True, 0.5, key_mask=mask)
    for algo in (0, 1):
        got = oracle.emul(q, k, v, True, 0.5, algo, 16, 52, 11, key_mask=mask)
        assert np.max(np.abs(got - want)) <= 1e-12
        assert np.all(got[0, :4] == 0.0)


def test_emul_format_trend_of_fig3():
    """FlashAttention vs baseline deviation falls as fraction bits grow."""
    q, k, v = _case(9, 2, 512, 32)
    scale = 1 / math.sqrt(32)
    dev = {}
    for fmt in ("bf16", "fp16", "fp32", "fp64"):
        mb, eb = oracle.FORMATS[fmt]
        base = oracle.emul(q, k, v, False, scale, 0, 64, mb, eb)
        tiled = oracle.emul(q, k, v, False, scale, 1, 64, mb, eb)
        dev[fmt] = np.max(np.abs(base - tiled))
    assert dev["bf16"] > dev["fp16"] > dev["fp32"] > dev["fp64"]
    assert dev["fp64"] <= 1e-13
    assert dev["bf16"] > 1e-3


def test_emul_row_subset_matches_full():
    q, k, v = _case(10, 3, 40, 8)
    full = oracle.emul(q, k, v, True, 0.3, 1, 8, 7, 8).reshape(-1, 8)
    rows = np.array([0, 5, 39, 40, 119])
    sub = oracle.emul(q, k, v, True, 0.3, 1, 8, 7, 8, rows=rows)
    assert np.array_equal(sub, full[rows])


def test_round_e5m2_matches_torch_float8_conversion():
    """The coarse format of the hand-worked rows below (2 fraction bits, 5
    exponent bits) is the E5M2 layout, which torch converts to with round to
    nearest even, subnormals and overflow to infinity."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("torch has no float8_e5m2")
    rng = np.random.default_rng(12)
    x32 = _wide_values(rng, 20000, -18, 17).astype(np.float32)   # subnormal E5M2 .. overflow
    want = torch.from_numpy(x32).to(torch.float8_e5m2).to(torch.float64).numpy()
    got = oracle.round_fmt(x32.astype(np.float64), 2, 5)
    assert np.array_equal(got, want)


def _golden_rows(golden_dir):
    import json
    import os
    with open(os.path.join(golden_dir, "emul_e5m2_rows.json")) as f:
        g = json.load(f)
    return g["format"]["mbits"], g["format"]["ebits"], g["cases"]


def _run_golden_row(case, mbits, ebits, plant=0):
    N = len(case["k"])
    q = np.full((1, N, 1), float(case["q"]))
    k = np.asarray(case["k"], dtype=np.float64).reshape(1, N, 1)
    v = np.asarray(case["v"], dtype=np.float64).reshape(1, N, 1)
    mask = None if case["mask"] is None else np.asarray(case["mask"], dtype=np.float64).reshape(1, N)
    out = oracle.emul(q, k, v, False, case["scale"], case["algo"], case["Bc"], mbits, ebits, key_mask=mask,
                      rows=[N - 1], plant=plant)
    return float(out[0, 0])


def test_emul_hand_worked_rows_e5m2(golden_dir):
    """Rows worked by hand, step by step, in the E5M2 layout (tests/golden/emul_e5m2_rows.json):
    both algorithms of the instrument, key blocks of 1 and 2, finite key masks.
    The oracle must give exactly the hand-worked output."""
    mb, eb, cases = _golden_rows(golden_dir)
    for case in cases:
        assert _run_golden_row(case, mb, eb) == case["O"], case["name"]


@pytest.mark.parametrize("site", sorted(oracle.EMUL_PLANTS))
def test_emul_planted_mistakes_fail_hand_worked_rows(golden_dir, site):
    """Every rounding site of the instrument is pinned: leaving one fl() out
    (Q, K or V not rounded first; the score, the mask sum, m - M, either exp,
    a*l, the row sum, the l update, a*o, the block's P V, the o update, the
    final division; the baseline's softmax or P V), rounding l only at the
    end, rounding P V after every key, rounding q.k after every term, or
    splitting the baseline softmax into three rounded ops changes the output
    of at least one hand-worked row."""
    mb, eb, cases = _golden_rows(golden_dir)
    plant = oracle.EMUL_PLANTS[site]
    changed = [c["name"] for c in cases if _run_golden_row(c, mb, eb, plant) != c["O"]]
    assert changed, f"planted mistake '{site}' is not caught by any hand-worked row"
