"""Number-format emulation on the GPU (attn_emul_fwd / attn_emul_round).

The emulation is the paper's numerical re-implementation ("Is Flash Attention
Stable?" §III, Fig. 2) used for its format sweep (§IV-A, Fig. 3) and its
block-size perturbations (§IV-B, Fig. 6).  Parity: the GPU rounding equals
the oracle's rounding bit for bit; emulated attention equals the oracle's
emulation (``oracle.emul``) to within a few units in the last place of the
format (the two sum their binary64 reductions in different orders and use
different libm exp, so a rounding to the format may rarely land on the other
neighbour) and, at binary64, the FP64 definition of attention.

With ETA_REPORT_DIR set, the format and block-width sweeps are written to
$ETA_REPORT_DIR/emul_sweeps.json.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

FMTS = ["bf16", "fp16", "tf32", "fp32", "fp64"]


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


def _wide_values(rng, n, lo, hi):
    e = rng.uniform(lo, hi, n)
    return np.where(rng.random(n) < 0.5, -1.0, 1.0) * np.exp2(e)


@pytest.mark.parametrize("fmt", FMTS)
def test_round_bitwise_equals_oracle(eta, fmt):
    mb, eb = eta.EMUL_FORMATS[fmt]
    rng = np.random.default_rng(11)
    x = np.concatenate([_wide_values(rng, 50000, -160, 140), [0.0, -0.0, np.inf, -np.inf, 65519.0, 65520.0]])
    want = oracle.round_fmt(x, mb, eb)
    got = eta.attn_emul_round(torch.from_numpy(x).cuda(), mb, eb).cpu().numpy()
    assert np.array_equal(got.view(np.int64), want.view(np.int64))


def _ulp_tol(fmt, ref):
    mb, _ = oracle.FORMATS[fmt]
    return 4.0 * 2.0 ** -mb * max(1.0, float(np.max(np.abs(ref))))


def _case(B, H, N, d, dtype, seed):
    q, k, v = workloads.make_qkv(B, H, N, d, dtype, seed)
    return q, k, v


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("algo,Bc", [(0, 1), (1, 1), (1, 16), (1, 64), (1, 200)])
@pytest.mark.parametrize("causal", [False, True])
def test_emul_matches_oracle_emulation(eta, fmt, algo, Bc, causal):
    B, H, N, d = 1, 2, 150, 32
    q, k, v = _case(B, H, N, d, "f32", seed=12)
    mb, eb = eta.EMUL_FORMATS[fmt]
    scale = float(np.float32(1 / math.sqrt(d)))   # the C ABI takes scale as float32
    got = eta.attn_emul_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale, algo, Bc, mb, eb).cpu().numpy()
    want = oracle.emul(q, k, v, causal, scale, algo, Bc, mb, eb)
    err = np.abs(got - want)
    if fmt == "fp64":
        assert err.max() <= 1e-12
        ref, _ = oracle.attn(q, k, v, causal, scale)
        assert np.max(np.abs(got - ref)) <= 1e-12
    else:
        assert err.max() <= _ulp_tol(fmt, want), err.max()
        assert np.mean(err == 0.0) >= 0.99


def test_emul_bf16_inputs_mask_and_row_subset(eta):
    B, H, N, d = 1, 4, 300, 64
    q, k, v = _case(B, H, N, d, "bf16", seed=13)
    mask = workloads.make_key_mask(B, H, N, 0.1, seed=13)       # heads h % 4 == 0: keys 0..3 masked
    rows = np.array([0, 1, 2, 3, 4, 299, 300, 777, 1199], dtype=np.int64)
    for algo, Bc in ((0, 1), (1, 64)):
        got = eta.attn_emul_fwd(q.cuda(), k.cuda(), v.cuda(), True, 0.125, algo, Bc, 7, 8, key_mask=mask.cuda(),
                                rows=torch.from_numpy(rows).cuda()).cpu().numpy()
        want = oracle.emul(q, k, v, True, 0.125, algo, Bc, 7, 8, key_mask=mask, rows=rows)
        assert np.max(np.abs(got - want)) <= _ulp_tol("bf16", want)
        assert np.all(got[:4] == 0.0)   # causal rows 0..3 of head 0 see only masked keys
    assert eta.attn_status() == 0


def test_emul_out_of_range_row_is_reported(eta):
    q, k, v = _case(1, 1, 64, 16, "f32", seed=14)
    rows = torch.tensor([0, 64, 5], dtype=torch.int64).cuda()     # 64 is out of range
    o = eta.attn_emul_fwd(q.cuda(), k.cuda(), v.cuda(), False, 0.25, 1, 16, 23, 8, rows=rows)
    assert eta.attn_status() == eta.ATTN_ERR_ARG
    assert eta.attn_status() == 0
    want = oracle.emul(q, k, v, False, 0.25, 1, 16, 23, 8, rows=np.array([0, 5]))
    got = o.cpu().numpy()[[0, 2]]
    assert np.max(np.abs(got - want)) <= _ulp_tol("fp32", want)


def test_emul_rejects_bad_arguments(eta):
    q, k, v = _case(1, 1, 32, 16, "f32", seed=15)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    for kwargs in ({"mbits": 0}, {"mbits": 53}, {"ebits": 1}, {"ebits": 12}, {"Bc": 0}, {"Bc": 5000}, {"algo": 2}):
        args = {"algo": 1, "Bc": 16, "mbits": 7, "ebits": 8}
        args.update(kwargs)
        with pytest.raises(eta.AttnError):
            eta.attn_emul_fwd(qc, kc, vc, False, 0.25, args["algo"], args["Bc"], args["mbits"], args["ebits"])


def test_format_and_block_sweeps(eta):
    """Fig. 3 (format sweep) and Fig. 6 (block width) at the length-sweep
    shape 1x8x4096x64, on 256 seeded rows; the FP64 definition is the golden
    value (Fig. 4)."""
    B, H, N, d = 1, 8, 4096, 64
    q, k, v = _case(B, H, N, d, "bf16", seed=0)
    scale = float(np.float32(1 / math.sqrt(d)))   # the C ABI takes scale as float32
    rows = workloads.sample_rows(B, H, N, 256 / (B * H * N), seed=16)
    rows_t = torch.from_numpy(np.asarray(rows, dtype=np.int64)).cuda()
    golden, _ = oracle.attn(q, k, v, False, scale, rows=rows)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()

    def run(algo, Bc, fmt):
        mb, eb = eta.EMUL_FORMATS[fmt]
        return eta.attn_emul_fwd(qc, kc, vc, False, scale, algo, Bc, mb, eb, rows=rows_t).cpu().numpy()

    report = {"shape": [B, H, N, d], "rows": len(rows), "format_sweep": [], "block_sweep": []}
    fa_vs_base = {}
    for fmt in FMTS:
        base = run(0, 1, fmt)
        tiled = run(1, 128, fmt)
        fa_vs_base[fmt] = float(np.max(np.abs(tiled - base)))
        report["format_sweep"].append({
            "format": fmt, "Bc": 128,
            "tiled_vs_baseline_max_abs": fa_vs_base[fmt],
            "tiled_vs_baseline_mean_abs": float(np.mean(np.abs(tiled - base))),
            "tiled_vs_golden_max_abs": float(np.max(np.abs(tiled - golden))),
            "baseline_vs_golden_max_abs": float(np.max(np.abs(base - golden))),
        })
    # more fraction bits, less deviation (the trend of Fig. 3)
    assert fa_vs_base["bf16"] > fa_vs_base["fp16"] > fa_vs_base["fp32"] > fa_vs_base["fp64"]
    assert fa_vs_base["fp64"] <= 1e-12
    base16 = run(0, 1, "bf16")
    by_bc = {}
    for Bc in (16, 32, 64, 128, 256, 512):
        tiled = run(1, Bc, "bf16")
        by_bc[Bc] = float(np.max(np.abs(tiled - base16)))
        report["block_sweep"].append({
            "format": "bf16", "Bc": Bc, "tiled_vs_baseline_max_abs": by_bc[Bc],
            "tiled_vs_baseline_mean_abs": float(np.mean(np.abs(tiled - base16))),
            "tiled_vs_golden_max_abs": float(np.max(np.abs(tiled - golden))),
        })
    # wider key blocks round the running state fewer times (the trend of Fig. 6c)
    assert by_bc[16] > by_bc[512]
    out = os.environ.get("ETA_REPORT_DIR")
    if out:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, "emul_sweeps.json"), "w") as f:
            json.dump(report, f, indent=1)
