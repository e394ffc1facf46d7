"""GPU parity of attn_fwd (through the C ABI) against the FP64 oracle.

Tolerances (max-abs on O): 1e-5 for float32 inputs, 2e-2 for bf16 inputs
with float32 accumulation.  LSE: |dLSE| <= 1e-5 * max(1, |LSE|) for float32
and 1e-3 + 2^-8 + 2e-6 * |LSE| for bf16 (derived in parity.py).
Fully masked rows must give O == 0 exactly and LSE == -inf, and no output
may be NaN.  Large configurations are checked on a seeded row subset that
always includes each head's first rows, last row and every fully masked row.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL_O, run_case  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


# ---------------- float32 path (CUDA cores) ----------------

def test_fp32_small_config(eta):
    """1 x 1 x 256 x 64, non-causal, seed 0: max-abs <= 1e-5."""
    w = workloads.WORKLOADS["fp32_1x1x256x64"]
    run_case(eta, w.B, w.H, w.N, w.d, "f32", w.causal)
    assert eta.attn_last_variant().startswith("simt_f32")


def test_fp32_worked_example(eta, golden_dir):
    """The tutorial's 5-score row embedded as a causal problem (q_i = e0,
    k_j = s_j e0, scale 1, d = 64 with zero padding): row i is the causal
    prefix of length i+1.  float32 holds 1000..1004 exactly."""
    import json, os
    g = json.load(open(os.path.join(golden_dir, "worked_example.json")))
    s = torch.tensor(g["scores"], dtype=torch.float32)
    vals = torch.tensor(g["values"], dtype=torch.float32)
    N, d = 5, 64
    q = torch.zeros(1, 1, N, d); q[..., 0] = 1.0
    k = torch.zeros(1, 1, N, d); k[0, 0, :, 0] = s
    v = torch.zeros(1, 1, N, d); v[0, 0, :, :2] = vals
    run_case(eta, 1, 1, N, d, "f32", True, scale=1.0, qkv=(q, k, v))
    o, lse = eta.attn_fwd(q.cuda(), k.cuda(), v.cuda(), True, 1.0)
    o = o.cpu().double()
    assert o[0, 0, 0, 0] == 2.0 and o[0, 0, 0, 1] == -1.0 and lse[0, 0, 0].item() == 1000.0
    e = math.e
    assert abs(o[0, 0, 1, 0].item() - 2 / (1 + e)) <= 1e-6
    assert abs(o[0, 0, 1, 1].item() - (3 * e - 1) / (1 + e)) <= 1e-6


@pytest.mark.parametrize("N", [1, 5, 63, 65, 129, 300])
@pytest.mark.parametrize("d", [17, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_tails(eta, N, d, causal):
    run_case(eta, 1, 2, N, d, "f32", causal, seed=N + d)


def test_fp32_masked_with_fully_masked_rows(eta):
    B, H, N, d = 1, 4, 200, 64
    mask = workloads.make_key_mask(B, H, N, 0.1, seed=3)
    mask[0, 1, :] = float("-inf")  # one head with no allowed key at all
    run_case(eta, B, H, N, d, "f32", False, mask=mask, seed=3)
    run_case(eta, B, H, N, d, "f32", True, mask=mask, seed=3)


# ---------------- bf16 path (tcgen05 tensor cores) ----------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Br", [64, 128])
@pytest.mark.parametrize("Bc", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_tiles_small(eta, d, Br, Bc, causal):
    """Every (Br, Bc) variant: several query groups, K/V ring wrap-around, ragged tail."""
    run_case(eta, 1, 3, 1000, d, "bf16", causal, Br=Br, Bc=Bc, seed=d + Bc + Br)
    assert f"_br{Br}_bc{Bc}_" in eta.attn_last_variant()


@pytest.mark.parametrize("N", [1, 5, 127, 128, 129, 255, 256, 257, 511, 513])
def test_bf16_tails(eta, N):
    run_case(eta, 2, 2, N, 128, "bf16", N % 2 == 1, seed=N)
    run_case(eta, 1, 2, N, 64, "bf16", N % 2 == 0, seed=N + 1)


@pytest.mark.parametrize("Bc", [64, 128, 256])
def test_bf16_masked(eta, Bc):
    B, H, N, d = 1, 4, 700, 128
    mask = workloads.make_key_mask(B, H, N, 0.05, seed=5)
    mask[0, 2, :] = float("-inf")
    run_case(eta, B, H, N, d, "bf16", True, Bc=Bc, mask=mask, seed=5)
    run_case(eta, B, H, N, d, "bf16", False, Bc=Bc, mask=mask, seed=5)


def test_bf16_config2_causal(eta):
    """4 x 16 x 1024 x 64 causal, every row."""
    w = workloads.WORKLOADS["bf16_causal_4x16x1024x64"]
    run_case(eta, w.B, w.H, w.N, w.d, "bf16", w.causal)
    assert eta.attn_last_variant().startswith("tc_bf16")


def test_bf16_config3_full_size(eta):
    """2 x 16 x 4096 x 128 non-causal at full size, in the benchmark's
    launch configuration; oracle on a seeded 1/32 row subset."""
    w = workloads.WORKLOADS["bf16_2x16x4096x128"]
    rows = workloads.sample_rows(w.B, w.H, w.N, 1 / 32, seed=0)
    run_case(eta, w.B, w.H, w.N, w.d, "bf16", w.causal, rows=rows)


def test_bf16_config5_adversarial(eta):
    """1 x 32 x 8192 x 128 causal, Q and K x30, 5% -inf key padding with
    fully masked rows; oracle on a seeded row subset plus every fully
    masked row."""
    w = workloads.WORKLOADS["bf16_causal_adv_1x32x8192x128"]
    q, k, v, mask = workloads.make_inputs(w)
    # fully masked rows under causality: row i of head h whose keys 0..i are all masked
    m = mask.numpy().reshape(w.B * w.H, w.N)
    extra = []
    for bh in range(w.B * w.H):
        allowed = np.cumsum(np.isfinite(m[bh]))
        extra += [bh * w.N + i for i in np.nonzero(allowed == 0)[0]]
    assert len(extra) > 0
    rows = workloads.sample_rows(w.B, w.H, w.N, 1 / 256, seed=0, extra=extra)
    run_case(eta, w.B, w.H, w.N, w.d, "bf16", w.causal, mask=mask, rows=rows, qkv=(q, k, v))


@pytest.mark.parametrize("Br,Bc", workloads.SWEEP_TILES)
def test_bf16_tile_sweep_config4(eta, Br, Bc):
    """The tile-size sweep shape: 1 x 8 x 4096 x 64 non-causal, every
    (Br, Bc) in {64,128} x {64,128,256}; oracle on a seeded row subset."""
    w = workloads.WORKLOADS["bf16_sweep_1x8xNx64"]
    rows = workloads.sample_rows(w.B, w.H, w.N, 1 / 64, seed=Br + Bc)
    run_case(eta, w.B, w.H, w.N, w.d, "bf16", w.causal, Br=Br, Bc=Bc, rows=rows)


@pytest.mark.parametrize("N", workloads.SWEEP_N)
def test_bf16_length_sweep_config4(eta, N):
    """The sequence-length sweep shape: 1 x 8 x N x 64, N = 128 .. 16384,
    default tiles; oracle on a seeded row subset (all rows for small N)."""
    w = workloads.WORKLOADS["bf16_sweep_1x8xNx64"]
    frac = 1.0 if N <= 1024 else 2048 / (w.B * w.H * N)
    rows = None if frac >= 1.0 else workloads.sample_rows(w.B, w.H, N, frac, seed=N)
    run_case(eta, w.B, w.H, N, w.d, "bf16", w.causal, rows=rows, seed=0)


def test_bf16_br_variants_agree(eta):
    """Rows are independent, so Br (rows per tile) must not change any
    result bit for a fixed Bc: the per-row arithmetic is the same."""
    q, k, v = workloads.make_qkv(1, 2, 777, 128, "bf16", 9)
    dev = torch.device("cuda")
    outs = []
    for br in (64, 128):
        o, l = eta.attn_fwd(q.to(dev), k.to(dev), v.to(dev), True, 1 / math.sqrt(128), br, 128)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


def test_guard_bands_untouched(eta):
    """O and LSE written in place inside larger buffers: the canary bands
    before and after them must be left alone (ragged N, causal)."""
    B, H, N, d = 1, 3, 333, 128
    q, k, v = workloads.make_qkv(B, H, N, d, "bf16", 11)
    dev = torch.device("cuda")
    n_o, n_l, pad = B * H * N * d, B * H * N, 4096
    obuf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((n_l + 2 * pad,), 7.0, dtype=torch.float32, device=dev)
    o = obuf[pad:pad + n_o].view(B, H, N, d)
    l = lbuf[pad:pad + n_l].view(B, H, N)
    eta.attn_fwd(q.to(dev), k.to(dev), v.to(dev), True, 1 / math.sqrt(d), out=o, lse=l)
    torch.cuda.synchronize()
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[pad + n_o:] == 7.0)
    assert torch.all(lbuf[:pad] == 7.0) and torch.all(lbuf[pad + n_l:] == 7.0)


def test_host_buffers_end_to_end(eta):
    """The host-memory path: pinned CPU tensors in, CPU tensors out."""
    q, k, v = workloads.make_qkv(1, 2, 256, 64, "bf16", 4)
    o, lse = eta.attn_fwd(q.pin_memory(), k.pin_memory(), v.pin_memory(), False, 0.125)
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    o_ref, _ = oracle.attn(q, k, v, False, 0.125)
    assert np.abs(o.double().numpy() - o_ref).max() <= 2e-2


def test_device_timeout_is_reported_and_recovered(eta):
    """A kernel whose wait can never complete gives up after its limit,
    records the timeout, and leaves the context usable."""
    assert eta.attn_status() == eta.ATTN_OK
    assert eta.attn_debug_wait_timeout(2000) == eta.ATTN_OK
    assert eta.attn_status() == eta.ATTN_ERR_DEVICE_TIMEOUT
    assert eta.attn_status() == eta.ATTN_OK   # cleared
    run_case(eta, 1, 1, 64, 64, "bf16", False)


def test_invalid_arguments_on_device(eta):
    q = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(eta.AttnError) as ei:
        eta.attn_fwd(q, q, q)
    assert ei.value.status == eta.ATTN_ERR_UNSUPPORTED


# ---------------- finite key-mask values (the mask enters S inside the MMA) ----------------

def _finite_mask(B, H, N, seed):
    """Additive key mask with finite values of every kind, not only 0 / -inf:
    ordinary values in [-6, 3), tiny ones (~1e-30), keys pushed down by ~200
    (their weights underflow), values not representable in bf16, and 5% -inf."""
    g = torch.Generator().manual_seed(seed)
    m = torch.empty(B, H, N).uniform_(-6.0, 3.0, generator=g)
    sel = torch.rand(B, H, N, generator=g)
    m = torch.where(sel < 0.05, torch.full_like(m, float("-inf")), m)
    m = torch.where((sel >= 0.05) & (sel < 0.10), m * 1e-30, m)
    m = torch.where((sel >= 0.10) & (sel < 0.15), m - 200.0, m)
    return m


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Br", [64, 128])
@pytest.mark.parametrize("Bc", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_finite_key_mask(eta, d, Br, Bc, causal):
    """Every (d, Br, Bc) variant with finite mask values: the tensor-core path
    adds mask / scale to q.k as three bf16 parts in one more MMA step, which
    must carry each float32 value (tiny, ordinary, large) to the scores."""
    B, H, N = 1, 3, 700
    mask = _finite_mask(B, H, N, seed=d + Bc + Br)
    run_case(eta, B, H, N, d, "bf16", causal, Br=Br, Bc=Bc, mask=mask, seed=d + Br)
    assert "_mask" in eta.attn_last_variant()


@pytest.mark.parametrize("scale", [0.0625, 0.25, 2.0])
def test_bf16_finite_key_mask_scales(eta, scale):
    """The MMA adds mask / scale; the softmax multiplies by scale again: the
    result must be scale * q.k + mask for small and large scales."""
    B, H, N, d = 1, 2, 513, 128
    mask = _finite_mask(B, H, N, seed=11)
    run_case(eta, B, H, N, d, "bf16", False, mask=mask, seed=12, scale=scale)
    run_case(eta, B, H, N, d, "bf16", True, mask=mask, seed=13, scale=scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Bc", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_zero_mask_bitwise_equals_no_mask(eta, d, Bc, causal):
    """A zero key mask adds exactly 0 to every score (the extra MMA step's
    products are all 0): O and LSE are bitwise those of the unmasked call."""
    q, k, v = (t.cuda() for t in workloads.make_qkv(1, 3, 1000, d, "bf16", d + Bc))
    zero = torch.zeros(1, 3, 1000, device="cuda")
    o0, l0 = eta.attn_fwd(q, k, v, causal, 1 / math.sqrt(d), 128, Bc)
    o1, l1 = eta.attn_fwd(q, k, v, causal, 1 / math.sqrt(d), 128, Bc, zero)
    torch.cuda.synchronize()
    assert "_mask" in eta.attn_last_variant()
    assert torch.equal(o0, o1)
    assert torch.equal(l0, l1)


def test_host_buffers_with_key_mask_match_device_call(eta):
    """The host-memory entry copies Q, K, V and the key mask into its
    workspace and runs the same kernel: O and LSE are bitwise those of the
    device-buffer call, and within tolerance of the oracle."""
    B, H, N, d = 1, 3, 450, 128
    q, k, v = workloads.make_qkv(B, H, N, d, "bf16", 21)
    mask = _finite_mask(B, H, N, seed=21)
    oh, lh = eta.attn_fwd(q.pin_memory(), k.pin_memory(), v.pin_memory(), True, 0.1, key_mask=mask.pin_memory())
    assert oh.device.type == "cpu" and lh.device.type == "cpu"
    od, ld = eta.attn_fwd(q.cuda(), k.cuda(), v.cuda(), True, 0.1, key_mask=mask.cuda())
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu())
    assert torch.equal(lh, ld.cpu())
    run_case(eta, B, H, N, d, "bf16", True, mask=mask, scale=0.1, qkv=(q, k, v))


# ---------------- long sequences (32-bit index arithmetic, many key tiles) ----------------

def test_bf16_long_sequence_noncausal(eta):
    """1 x 2 x 131072 x 64 non-causal (1024 key tiles per row, split tail);
    oracle on a seeded row sample with each head's first and last rows."""
    B, H, N, d = 1, 2, 131072, 64
    rows = workloads.sample_rows(B, H, N, 48 / (B * H * N), seed=1)
    run_case(eta, B, H, N, d, "bf16", False, rows=rows, seed=31)


def test_bf16_long_sequence_causal_masked(eta):
    """1 x 1 x 65536 x 128 causal with finite key-mask values and -inf keys."""
    B, H, N, d = 1, 1, 65536, 128
    mask = _finite_mask(B, H, N, seed=32)
    rows = workloads.sample_rows(B, H, N, 48 / (B * H * N), seed=2, extra=[N - 2, N // 2])
    run_case(eta, B, H, N, d, "bf16", True, mask=mask, rows=rows, seed=32)


@pytest.mark.parametrize("N", [1, 2, 3, 31, 127, 129, 255, 257])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_finite_key_mask_ragged(eta, N, d):
    """Ragged lengths with finite mask values: the mask operand of the last
    K tile holds the mask for keys < N only, and zeros past N."""
    B, H = 1, 2
    mask = _finite_mask(B, H, N, seed=N + d)
    run_case(eta, B, H, N, d, "bf16", N % 2 == 1, mask=mask, seed=N + d)
    run_case(eta, B, H, N, d, "bf16", N % 2 == 0, mask=mask, seed=N + d + 1)
