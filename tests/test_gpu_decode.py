"""Decode with a key/value cache (attn_decode_fwd) against the FP64 oracle.

The oracle computes ordinary attention over equal-length Q and K.  A decode
problem (Nq new query rows at positions Nk - Nq .. Nk - 1 of an Nk-long
sequence) is embedded in it exactly: the Nq rows are placed at the end of an
Nk-row query tensor (the other rows are zeros and are not evaluated), and the
oracle evaluates only those rows.  With the oracle's top-left causal rule,
row Nk - Nq + i then sees keys j <= Nk - Nq + i, which is the decode rule.

Tolerances are those of the forward tests: bf16 max-abs 2e-2 on O, float32
1e-5; LSE 1e-3 + 2e-6|LSE| (bf16) and 1e-5 max(1, |LSE|) (float32).
"""
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


def _oracle_decode(q, k, v, causal, scale, mask=None):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    L = max(Nk, Nq)   # non-causal rows may outnumber the keys: pad with masked keys
    qfull = torch.zeros((B, H, L, d), dtype=torch.float64)
    qfull[:, :, L - Nq:, :] = q.double()
    kf = torch.zeros((B, H, L, d), dtype=torch.float64)
    vf = torch.zeros((B, H, L, d), dtype=torch.float64)
    kf[:, :, :Nk] = k.double()
    vf[:, :, :Nk] = v.double()
    mf = torch.full((B, H, L), -float("inf"), dtype=torch.float64)
    mf[:, :, :Nk] = 0.0 if mask is None else mask.double()
    rows = np.array([bh * L + L - Nq + i for bh in range(B * H) for i in range(Nq)], dtype=np.int64)
    o, lse = oracle.attn(qfull, kf, vf, causal, scale, key_mask=mf, rows=rows)
    return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)


def _check(eta, q, k, v, causal, mask=None, dtype="bf16"):
    d = q.shape[-1]
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = eta.attn_decode_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale,
                                 key_mask=mask.cuda() if mask is not None else None)
    o_ref, lse_ref = _oracle_decode(q, k, v, causal, scale, mask)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    assert not np.isnan(og).any()
    tol = 2e-2 if dtype == "bf16" else 1e-5
    assert np.max(np.abs(og - o_ref)) <= tol
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), inf_ref)
    assert np.all(og[inf_ref] == 0.0)
    fin = ~inf_ref
    ltol = 1e-3 + 2e-6 * np.abs(lse_ref[fin]) if dtype == "bf16" else 1e-5 * np.maximum(1.0, np.abs(lse_ref[fin]))
    assert np.all(np.abs(lg[fin] - lse_ref[fin]) <= ltol)


def _qkv(B, H, Nq, Nk, d, dtype, seed):
    q, _, _ = workloads.make_qkv(B, H, Nq, d, dtype, seed)
    _, k, v = workloads.make_qkv(B, H, Nk, d, dtype, seed + 100)
    return q, k, v


@pytest.mark.parametrize("Nq", [1, 3, 8])
@pytest.mark.parametrize("Nk", [1, 31, 257, 4097])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_bf16_lengths(eta, Nq, Nk, causal):
    if causal and Nq > Nk:
        pytest.skip("causal decoding needs Nq <= Nk")
    q, k, v = _qkv(2, 3, Nq, Nk, 128, "bf16", seed=Nq * 7 + Nk)
    _check(eta, q, k, v, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
def test_decode_head_dims_f32(eta, d):
    q, k, v = _qkv(1, 4, 4, 700, d, "f32", seed=d)
    _check(eta, q, k, v, True, dtype="f32")


def test_decode_key_mask_and_fully_masked_rows(eta):
    B, H, Nq, Nk, d = 1, 4, 2, 1000, 64
    q, k, v = _qkv(B, H, Nq, Nk, d, "bf16", seed=5)
    mask = workloads.make_key_mask(B, H, Nk, 0.05, seed=5)
    mask[0, 1, :] = -float("inf")             # head 1: every key masked
    _check(eta, q, k, v, False, mask=mask)


def test_decode_long_cache_bf16(eta):
    """One new token per head against a 32768-long cache (the bulk decode shape)."""
    q, k, v = _qkv(1, 4, 1, 32768, 128, "bf16", seed=9)
    _check(eta, q, k, v, True)


def test_decode_rejects_unsupported(eta):
    q, k, v = _qkv(1, 1, 9, 64, 64, "bf16", seed=1)
    with pytest.raises(eta.AttnError):
        eta.attn_decode_fwd(q.cuda(), k.cuda(), v.cuda(), False)          # Nq > 8
    q2, k2, v2 = _qkv(1, 1, 2, 64, 80, "bf16", seed=2)
    with pytest.raises(eta.AttnError):
        eta.attn_decode_fwd(q2.cuda(), k2.cuda(), v2.cuda(), False)       # d not a multiple of 32
    q3, k3, v3 = _qkv(1, 1, 4, 3, 64, "bf16", seed=3)
    with pytest.raises(eta.AttnError):
        eta.attn_decode_fwd(q3.cuda(), k3.cuda(), v3.cuda(), True)        # causal with Nq > Nk
    q4, k4, v4 = _qkv(1, 2, 2, 64, 64, "bf16", seed=4)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(eta.AttnError):
        eta.attn_decode_fwd(q4.cuda(), k4.cuda(), v4.cuda(), False, workspace=small)


def test_decode_many_stage_rounds(eta):
    """A 262144-long cache on one head: every CTA streams 64 groups of keys
    through its ring, so each stage is refilled many times."""
    q, k, v = _qkv(1, 1, 1, 262144, 64, "bf16", seed=11)
    _check(eta, q, k, v, True)
