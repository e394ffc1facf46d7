"""Deviation sweeps in the manner of "Is Flash Attention Stable?":

* Fig. 4: the tiled forward and the materialising baseline, each against the
  FP64 golden value (here the FP64 oracle), at bf16;
* Fig. 5: deviation versus sequence length at fixed tile sizes;
* Fig. 6b/6c: deviation versus tile size (square and non-square tiles).

Deviation is measured with the library's own attn_deviation (max-abs,
Wasserstein-1 via the device sort, mean/std of |d|) on a seeded subset of
query rows, cross-checked against the oracle's CPU deviation.  Every cell
must meet the bf16 tolerance (max-abs <= 2e-2).  With ETA_REPORT_DIR set, the
table is written to $ETA_REPORT_DIR/deviation_sweeps.json.
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
TOL = 2e-2
ROWS_PER_CELL = 1024


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


@pytest.fixture(scope="module")
def report():
    table = []
    yield table
    out = os.environ.get("ETA_REPORT_DIR")
    if out:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, "deviation_sweeps.json"), "w") as f:
            json.dump(table, f, indent=1)


def _rows(B, H, N, seed):
    total = B * H * N
    if total <= ROWS_PER_CELL:
        return np.arange(total)
    g = torch.Generator().manual_seed(seed)
    return np.sort(torch.randperm(total, generator=g)[:ROWS_PER_CELL].numpy())


def _dev(eta, out_rows, golden):
    d = eta.attn_deviation(out_rows.reshape(-1), torch.from_numpy(golden.reshape(-1)).cuda())
    c = oracle.deviation(out_rows.double().cpu().numpy(), golden)
    assert math.isclose(d["max_abs"], c["max_abs"], rel_tol=1e-12, abs_tol=1e-15)
    assert math.isclose(d["w1"], c["w1"], rel_tol=1e-9, abs_tol=1e-15)
    return d


def _cell(eta, report, label, w, N, Br, Bc, with_naive=False, seed=0):
    q, k, v, mask = workloads.make_inputs(w, seed=seed, N=N)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = mask.to(dev) if mask is not None else None
    rows = _rows(w.B, w.H, N, seed + N + Br + Bc)
    golden, _ = oracle.attn(q, k, v, w.causal, w.scale, key_mask=mask, rows=rows)
    o, _ = eta.attn_fwd(qd, kd, vd, w.causal, w.scale, Br, Bc, md)
    o_rows = o.reshape(-1, w.d)[torch.from_numpy(rows).to(dev)]
    d_fa = _dev(eta, o_rows, golden)
    entry = {"sweep": label, "workload": w.name, "N": N, "Br": Br or 128, "Bc": Bc or 128,
             "rows": int(len(rows)), "tiled": {k2: d_fa[k2] for k2 in ("max_abs", "w1", "mean_abs", "std_abs")}}
    assert d_fa["max_abs"] <= TOL
    if with_naive:
        on, _ = eta.attn_naive_fwd(qd, kd, vd, w.causal, w.scale, md)
        n_rows = on.reshape(-1, w.d)[torch.from_numpy(rows).to(dev)]
        d_nv = _dev(eta, n_rows, golden)
        entry["baseline"] = {k2: d_nv[k2] for k2 in ("max_abs", "w1", "mean_abs", "std_abs")}
    report.append(entry)


@pytest.mark.parametrize("N", workloads.SWEEP_N)
def test_length_sweep(eta, report, N):
    """[Fig. 5] 1 x 8 x N x 64 bf16, tiles fixed at (128, 128)."""
    w = workloads.WORKLOADS["bf16_sweep_1x8xNx64"]
    _cell(eta, report, "length", w, N, 128, 128, with_naive=(N <= 8192))


@pytest.mark.parametrize("Br,Bc", workloads.SWEEP_TILES)
def test_tile_sweep(eta, report, Br, Bc):
    """[Fig. 6b/6c] 1 x 8 x 4096 x 64 bf16, (Br, Bc) in {64,128} x {64,128,256}."""
    w = workloads.WORKLOADS["bf16_sweep_1x8xNx64"]
    _cell(eta, report, "tile", w, 4096, Br, Bc)


@pytest.mark.parametrize("name", ["bf16_causal_4x16x1024x64", "bf16_2x16x4096x128",
                                  "bf16_causal_adv_1x32x8192x128"])
def test_golden_comparison(eta, report, name):
    """[Fig. 4] tiled forward and materialising baseline vs the FP64 golden."""
    w = workloads.WORKLOADS[name]
    _cell(eta, report, "golden", w, w.N, 0, 0, with_naive=True)
