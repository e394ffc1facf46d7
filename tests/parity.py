"""Shared parity check for the GPU forward tests (not collected by pytest).

run_case() runs attn_fwd through the C ABI on seeded (or given) inputs and
compares O and LSE with the FP64 oracle, element by element: max-abs on O of
1e-5 for float32 inputs and 2e-2 for bf16 inputs with float32 accumulation.
LSE: |dLSE| <= 1e-5 * max(1, |LSE|) for float32 (float32 rounding of the
scaled scores).  For bf16, |dLSE| <= 1e-3 + 2^-8 + 2e-6 * |LSE|.  The
2e-6 * |LSE| term covers float32 scores up to ~1e4.  The 2^-8 term covers
the denominator: it sums the p rounded to bf16 (the weights O applies), each
within a relative 2^-8 of p, so its log is within ln(1 + 2^-8) < 2^-8 of the
exact one.  Fully masked rows must give O == 0 exactly and LSE == -inf, and
no output may be NaN.
"""
import math

import numpy as np
import torch

import oracle
import workloads

TOL_O = {"f32": 1e-5, "bf16": 2e-2}


def _lse_tol(dtype, ref):
    a = np.abs(np.where(np.isfinite(ref), ref, 0.0))
    return 1e-5 * np.maximum(1.0, a) if dtype == "f32" else 1e-3 + 2.0 ** -8 + 2e-6 * a


def run_case(eta, B, H, N, d, dtype, causal, Br=0, Bc=0, mask=None, qk_scale=1.0, seed=0, rows=None,
             scale=None, qkv=None):
    if qkv is None:
        q, k, v = workloads.make_qkv(B, H, N, d, dtype, seed, qk_scale)
    else:
        q, k, v = qkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dev = torch.device("cuda")
    o, lse = eta.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal, scale, Br, Bc,
                          mask.to(dev) if mask is not None else None)
    torch.cuda.synchronize()
    assert eta.attn_status() == eta.ATTN_OK
    o_ref, lse_ref = oracle.attn(q, k, v, causal, scale, key_mask=mask, rows=rows)
    og = o.double().cpu().numpy().reshape(-1, d)
    lg = lse.double().cpu().numpy().reshape(-1)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    o_ref = o_ref.reshape(-1, d)
    lse_ref = lse_ref.reshape(-1)
    assert not np.isnan(og).any() and not np.isnan(lg).any()
    err = np.abs(og - o_ref).max()
    assert err <= TOL_O[dtype], f"max|dO| = {err}"
    inf_ref = np.isneginf(lse_ref)
    np.testing.assert_array_equal(np.isneginf(lg), inf_ref)
    assert np.all(og[inf_ref] == 0.0)
    fin = ~inf_ref
    lerr = np.abs(lg[fin] - lse_ref[fin])
    assert np.all(lerr <= _lse_tol(dtype, lse_ref[fin])), f"max|dLSE| = {lerr.max()}"
    return err
