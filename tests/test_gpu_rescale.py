"""GPU parity of the tensor-core forward where its rescaling shortcuts decide.

The kernel keeps each row's online-softmax state as the yadro-code.ru
FlashAttention tutorial describes it (a running maximum, a running
denominator and an unnormalised accumulator, brought to a common maximum
when a block with a larger one arrives), with two shortcuts that are exact up
to rounding because O / l does not depend on the reference point:

- the reference maximum moves only to a tile maximum more than 8 (log2
  units) above it, so a tile is exponentiated against a reference that may
  lie below its maximum, every p stays below 2^8, and O is rescaled only when
  the reference moves;
- the row's denominator is the sum of the bf16-rounded p that P V applies.

These tests put row scores just below and just above the limit, on every
(d, Br, Bc) variant, causal and not, through exact embeddings (q = e0 plus a
small second component, k_j = s_j e0 plus a small second component, scale =
ln 2 so that a score is its own log2-domain value).  They also run the
adversarial workload's generator (Q and K x30, -inf key padding, fully
masked rows) through every variant and through the K/V-split cluster tail,
and run CTAs through several work units repeatedly: the results must be
bitwise the same every time.
Bar: the forward's bf16 tolerance against the FP64 oracle (O max-abs 2e-2;
LSE 1e-3 + 2^-8 + 2e-6 |LSE|; fully masked rows O = 0, LSE = -inf).
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import run_case

pytestmark = pytest.mark.gpu

VARIANTS = [(d, br, bc) for d in (64, 128) for br in (64, 128) for bc in (64, 128, 256)]
SCALE = float(np.float32(math.log(2.0)))   # score s * scale * log2(e) = s (to float32 rounding)


@pytest.fixture(scope="module")
def eta():
    import exact_tiled_attention_17_gb300 as m
    return m


def _embedding(N, d, Bc, high, low, H=2, seed=0):
    """q_i = e0 + c_i e1, k_j = x_j e0 + r_j e1 (bf16-exact), V ~ N(0, 1).

    Key tile t = keys [t*Bc, (t+1)*Bc): one key (its column moves from tile to
    tile) at score high(t), the others at low(t).  c_i in {-1, 0, 1}, r_j in
    {-0.25, 0, 0.25}, so a row's scores differ from x_j by at most 0.25."""
    x = np.empty(N)
    for t in range(-(-N // Bc)):
        j0, j1 = t * Bc, min(N, (t + 1) * Bc)
        x[j0:j1] = low(t)
        hk = j0 + (37 * t + 5) % Bc
        if hk < j1:
            x[hk] = high(t)
    q = torch.zeros(1, H, N, d)
    k = torch.zeros(1, H, N, d)
    q[..., 0] = 1.0
    q[..., 1] = torch.tensor([(i % 3) - 1.0 for i in range(N)])
    k[..., 0] = torch.from_numpy(x).float()
    k[..., 1] = torch.tensor([0.25 * ((j % 3) - 1) for j in range(N)])
    qb, kb = q.to(torch.bfloat16), k.to(torch.bfloat16)
    assert torch.equal(qb.float(), q) and torch.equal(kb.float(), k), "embedding must be bf16-exact"
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(1, H, N, d, generator=g).to(torch.bfloat16)
    return qb, kb, v


# plateau: the first tile's keys at 0 set the reference; every later tile has
# one key at `delta` above it and the rest at 0.
#   delta 15.5: a tile's sum stays below 2^16 (no redo); 16.5: above (redo).
#   delta 7 / 9: below / above the 256-column variant's move limit of 8.
@pytest.mark.parametrize("delta", [7.0, 9.0, 15.5, 16.5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Br,Bc", VARIANTS)
def test_reference_plateau_around_limits(eta, d, Br, Bc, causal, delta):
    N = 1000
    qkv = _embedding(N, d, Bc, high=lambda t: 0.0 if t == 0 else delta, low=lambda t: 0.0, seed=int(delta))
    run_case(eta, 1, 2, N, d, "bf16", causal, Br=Br, Bc=Bc, scale=SCALE, qkv=qkv)
    assert f"_br{Br}_bc{Bc}_" in eta.attn_last_variant()


# staircase: tile t's high key at delta * (t mod 8), the rest 20 below it.
#   delta 17: every step passes 2^16 (a redo per tile); delta 15: every other
#   step does (the reference moves on alternate tiles).
@pytest.mark.parametrize("delta", [15.0, 17.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Br,Bc", VARIANTS)
def test_reference_staircase(eta, d, Br, Bc, causal, delta):
    N = 1000
    qkv = _embedding(N, d, Bc, high=lambda t: delta * (t % 8), low=lambda t: delta * (t % 8) - 20.0,
                     seed=int(delta) + 1)
    run_case(eta, 1, 2, N, d, "bf16", causal, Br=Br, Bc=Bc, scale=SCALE, qkv=qkv)


def _adversarial(B, H, N, d, seed, all_masked_head=None):
    q, k, v = workloads.make_qkv(B, H, N, d, "bf16", seed, qk_scale=30.0)
    mask = workloads.make_key_mask(B, H, N, 0.05, seed=seed)
    if all_masked_head is not None:
        mask[0, all_masked_head, :] = float("-inf")
    return q, k, v, mask


def _fully_masked_rows(mask, causal):
    m = mask.numpy().reshape(-1, mask.shape[-1])
    out = []
    for bh in range(m.shape[0]):
        allowed = np.cumsum(np.isfinite(m[bh])) if causal else np.full(m.shape[1], np.isfinite(m[bh]).sum())
        out += [bh * m.shape[1] + i for i in np.nonzero(allowed == 0)[0]]
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Br,Bc", VARIANTS)
def test_adversarial_logits_every_variant(eta, d, Br, Bc, causal):
    """The adversarial workload's generator at 1 x 4 x 1000: Q, K x30 (scaled
    scores in the thousands), 5% -inf key padding, keys 0..3 masked in head
    0 (causal rows 0..3 fully masked) and head 1 masked whole."""
    B, H, N = 1, 4, 1000
    q, k, v, mask = _adversarial(B, H, N, d, seed=d + Br + Bc, all_masked_head=1)
    assert len(_fully_masked_rows(mask, causal)) > 0
    run_case(eta, B, H, N, d, "bf16", causal, Br=Br, Bc=Bc, mask=mask, qkv=(q, k, v))
    assert f"_br{Br}_bc{Bc}_" in eta.attn_last_variant()


def _heads_for_split(nsm, num_qg, split, nkv, after_full_rounds):
    """Heads H (B = 1) whose items (H * num_qg of them) leave R = items mod nsm
    past the last full round with split * R <= nsm and, below 8 parts,
    2 * split * R > nsm: the launcher then splits each of those R items into
    `split` parts.  after_full_rounds: items = nsm + R (a full round of whole
    items first), else items = R (the launch is the split tail alone)."""
    if nsm % split or split > nkv:
        return None
    for R in range(1, nsm + 1):
        if split * R > nsm:
            break
        if split < 8 and 2 * split * R <= nsm:
            continue
        items = nsm + R if after_full_rounds else R
        if items % num_qg == 0:
            return items // num_qg
    return None


@pytest.mark.parametrize("split,after_full_rounds", [(2, True), (2, False), (4, False), (8, False)])
@pytest.mark.parametrize("d,Bc", [(128, 128), (64, 128), (128, 64), (64, 256)])
def test_adversarial_logits_split_tail(eta, d, Bc, split, after_full_rounds):
    """Non-causal items past the last full round are split along K/V over the
    CTAs of a cluster and merged with the tiles' rescale rule.  Heads are
    chosen from the SM count so that the tail splits into 2, 4 or 8 parts,
    after a full round of whole items or as the whole launch; one head has
    every key masked (each part's maximum is -inf)."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    N, Br = 1000, 128
    nq = 2 if 2 * (Bc + d) <= 512 else 1
    num_qg = -(-N // (nq * Br))
    H = _heads_for_split(nsm, num_qg, split, -(-N // Bc), after_full_rounds)
    if H is None:
        pytest.skip(f"no head count splits the tail {split} ways on {nsm} SMs with Bc={Bc}")
    q, k, v, mask = _adversarial(1, H, N, d, seed=split + d, all_masked_head=2 % H)
    extra = _fully_masked_rows(mask, False)
    rows = workloads.sample_rows(1, H, N, 1 / 16, seed=split, extra=extra)
    run_case(eta, 1, H, N, d, "bf16", False, Br=Br, Bc=Bc, mask=mask, rows=rows, qkv=(q, k, v))
    assert f"_kvsplit{split}" in eta.attn_last_variant()
    # the same heads unmasked, N(0, 1) inputs
    run_case(eta, 1, H, N, d, "bf16", False, Br=Br, Bc=Bc, rows=rows, seed=split)
    assert f"_kvsplit{split}" in eta.attn_last_variant()


@pytest.mark.parametrize("mask_kind", ["none", "zero", "padding"])
@pytest.mark.parametrize("d,Bc", [(64, 128), (128, 128), (64, 64)])
def test_repeated_runs_bitwise_identical(eta, d, Bc, mask_kind):
    """x30 logits (the reference moves often) with every CTA running at least
    two work units, repeated: every run bitwise equal to the first, and the
    first within tolerance of the oracle.  (A row maximum read from a
    tensor-memory load before the load has completed made this vary between
    runs.)"""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    N, Br = 1000, 128
    nq = 2 if 2 * (Bc + d) <= 512 else 1
    num_qg = -(-N // (nq * Br))
    H = -(-2 * nsm // num_qg)
    q, k, v, mask = _adversarial(1, H, N, d, seed=d + Bc, all_masked_head=2)
    if mask_kind == "zero":
        mask = torch.zeros_like(mask)
    elif mask_kind == "none":
        mask = None
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = mask.to(dev) if mask is not None else None
    scale = 1.0 / math.sqrt(d)
    first = None
    for rep in range(6):
        o, lse = eta.attn_fwd(qd, kd, vd, False, scale, Br, Bc, md)
        torch.cuda.synchronize()
        assert eta.attn_status() == eta.ATTN_OK
        if first is None:
            first = (o.clone(), lse.clone())
        else:
            assert torch.equal(o, first[0]), f"run {rep}: O differs from the first run"
            assert torch.equal(lse, first[1]), f"run {rep}: LSE differs from the first run"
    extra = _fully_masked_rows(mask, False) if mask is not None else []
    rows = workloads.sample_rows(1, H, N, 1 / 32, seed=d, extra=extra)
    run_case(eta, 1, H, N, d, "bf16", False, Br=Br, Bc=Bc, mask=mask, rows=rows, qkv=(q, k, v))


@pytest.mark.parametrize("d", [64, 128])
def test_masked_split_tail_two_batches(eta, d):
    """B = 2 with finite key-mask values and -inf keys, heads chosen so that
    the non-causal tail splits along K/V: each (batch, head) reads its own
    mask row in every part."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    N, Br, Bc = 1000, 128, 128
    num_qg = -(-N // (2 * Br))
    H = _heads_for_split(nsm, num_qg, 2, -(-N // Bc), True)
    if H is None or H % 2:
        pytest.skip("no even head count splits the tail 2 ways on this GPU")
    B, Hh = 2, H // 2
    g = torch.Generator().manual_seed(d)
    mask = torch.empty(B, Hh, N).uniform_(-6.0, 3.0, generator=g)
    sel = torch.rand(B, Hh, N, generator=g)
    mask = torch.where(sel < 0.05, torch.full_like(mask, float("-inf")), mask)
    rows = workloads.sample_rows(B, Hh, N, 1 / 16, seed=d)
    run_case(eta, B, Hh, N, d, "bf16", False, Br=Br, Bc=Bc, mask=mask, rows=rows, seed=d)
    assert "_kvsplit2" in eta.attn_last_variant()


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_split_tail_writes_every_element(eta, d, split):
    """Every part of a split item merges and stores its own share of O's
    32-column chunks (part 0 also the LSE).  With O and LSE filled with NaN
    before the call, every element comes back finite, and sampled rows match
    the oracle."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    N, Br, Bc = 1000, 128, 128
    num_qg = -(-N // (2 * Br))
    H = _heads_for_split(nsm, num_qg, split, -(-N // Bc), False)
    if H is None:
        pytest.skip(f"no head count splits the tail {split} ways on {nsm} SMs")
    q, k, v = workloads.make_qkv(1, H, N, d, "bf16", seed=40 + split)
    dev = torch.device("cuda")
    o = torch.full((1, H, N, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((1, H, N), float("nan"), dtype=torch.float32, device=dev)
    eta.attn_fwd(q.to(dev), k.to(dev), v.to(dev), False, 1.0 / math.sqrt(d), Br, Bc, None, out=o, lse=lse)
    torch.cuda.synchronize()
    assert eta.attn_status() == eta.ATTN_OK
    assert f"_kvsplit{split}" in eta.attn_last_variant()
    assert not torch.isnan(o).any(), "an O element was not written"
    assert not torch.isnan(lse).any(), "an LSE element was not written"
    rows = workloads.sample_rows(1, H, N, 1 / 16, seed=split)
    run_case(eta, 1, H, N, d, "bf16", False, Br=Br, Bc=Bc, rows=rows, qkv=(q, k, v))
    assert f"_kvsplit{split}" in eta.attn_last_variant()


def test_dependent_launch_chain_matches_synchronised_calls(eta):
    """The forward, backward and decode kernels are programmatic dependent
    launches: each waits for the grid before it in the stream before it
    touches global memory.  A chain of calls that each read the previous
    call's output, enqueued back to back, gives bitwise the same O, LSE, dK
    and dV as the same calls with a synchronize after each (dQ, reduced with
    float atomics in any order, within rounding), and the chain's first
    output matches the oracle."""
    B, H, N, d = 1, 4, 1000, 128
    q, k, v = workloads.make_qkv(B, H, N, d, "bf16", seed=77)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    scale = 1.0 / math.sqrt(d)

    def chain(sync):
        def s():
            if sync:
                torch.cuda.synchronize()
        o1, l1 = eta.attn_fwd(qd, kd, vd, False, scale)
        s()
        o2, l2 = eta.attn_fwd(o1, kd, vd, True, scale)     # the last output as the queries
        s()
        o3, l3 = eta.attn_fwd(o2, kd, o1, False, scale)    # and as the values
        s()
        dq, dk, dv = eta.attn_bwd(o2, kd, o1, o3, o2, l3, False, scale)
        s()
        od, ld = eta.attn_decode_fwd(dk[:, :, N - 4:].contiguous(), kd, dv, True, scale)
        s()
        o4, l4 = eta.attn_fwd(dv, dk, o3, False, scale)
        torch.cuda.synchronize()
        assert eta.attn_status() == eta.ATTN_OK
        return [t.clone() for t in (o1, l1, o2, l2, o3, l3, dq, dk, dv, od, ld, o4, l4)]

    a = chain(False)
    b = chain(True)
    names = ["o1", "l1", "o2", "l2", "o3", "l3", "dq", "dk", "dv", "od", "ld", "o4", "l4"]
    for name, x, y in zip(names, a, b):
        if name == "dq":
            assert torch.allclose(x.float(), y.float(), rtol=0, atol=1e-2 * max(1.0, y.float().abs().max().item()))
        else:
            assert torch.equal(x, y), f"{name} differs between the chained and the synchronised calls"
    rows = workloads.sample_rows(B, H, N, 1 / 16, seed=77)
    run_case(eta, B, H, N, d, "bf16", False, rows=rows, qkv=(q, k, v))
