"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random numbers,
scales them, rounds them to the storage dtype and builds masks.  Both the
CUDA path's callers and the oracle's callers take their inputs from here, so
both sides see bit-identical values.

Recipe (every workload): Q, K, V are drawn, in that order, as float32
N(0, 1) samples from ``torch.Generator(device="cpu").manual_seed(seed)``,
optionally multiplied by a logit-scale factor (Q and K only), then rounded
to the storage dtype with round-to-nearest-even.  Layout is [B][H][N][d],
contiguous.  scale = 1/sqrt(d).

The five workloads are the paper's forward-pass micro-benchmark shapes
restated for one GB300 ("Is Flash Attention Stable?" §IV, random Q/K/V
inputs with identical inputs fed to every implementation; the sequence-
length sweep of its Fig. 5 and the tile-size sweep of its Fig. 6), plus an
adversarial large-logit case with a key-padding mask that exercises the
true -inf masking the aicompass.dev post on FlashInfer's -50,000 sentinel
is about.  There is no dataset: the paper's text-to-image training data is
not used and is not needed for the forward pass.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dtype: str                 # "f32" or "bf16": storage and input dtype
    qk_scale: float = 1.0      # Q and K are multiplied by this after drawing
    mask_frac: float = 0.0     # fraction of keys masked with -inf (key padding)
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved for causal: the two contractions only."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def with_n(self, N: int) -> "Workload":
        return Workload(self.name, self.B, self.H, N, self.d, self.causal, self.dtype,
                        self.qk_scale, self.mask_frac, self.note)


WORKLOADS = {
    "fp32_1x1x256x64": Workload("fp32_1x1x256x64", 1, 1, 256, 64, False, "f32",
                                note="small FP32 case the oracle finishes in seconds"),
    "bf16_causal_4x16x1024x64": Workload("bf16_causal_4x16x1024x64", 4, 16, 1024, 64, True, "bf16"),
    "bf16_2x16x4096x128": Workload("bf16_2x16x4096x128", 2, 16, 4096, 128, False, "bf16",
                                   note="image-token-like self-attention; the headline throughput shape"),
    "bf16_sweep_1x8xNx64": Workload("bf16_sweep_1x8xNx64", 1, 8, 4096, 64, False, "bf16",
                                    note="N swept over 128..16384 by powers of two; tiles swept at N=4096"),
    "bf16_causal_adv_1x32x8192x128": Workload("bf16_causal_adv_1x32x8192x128", 1, 32, 8192, 128, True,
                                              "bf16", qk_scale=30.0, mask_frac=0.05,
                                              note="Q,K x30 logits, 5% -inf key padding, fully masked rows"),
}

SWEEP_N = [128 * 2 ** i for i in range(8)]          # 128 .. 16384
SWEEP_TILES = [(br, bc) for br in (64, 128) for bc in (64, 128, 256)]

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_qkv(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
             qk_scale: float = 1.0):
    """Q, K, V as CPU tensors of the storage dtype, [B][H][N][d], contiguous."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    t = TORCH_DTYPE[dtype]
    return q.to(t).contiguous(), k.to(t).contiguous(), v.to(t).contiguous()


def make_grad_out(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0):
    """Upstream gradient dO for the backward pass: float32 N(0, 1) from its own
    stream (seed + 3, so it does not disturb Q/K/V or the mask), rounded to
    the storage dtype, [B][H][N][d] contiguous on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(seed + 3)
    do = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    return do.to(TORCH_DTYPE[dtype]).contiguous()


def make_block_mask(B: int, H: int, N: int, density: float = 0.5, seed: int = 0, pattern: str = "random",
                    window: int = 2, block: int = 128):
    """Block mask for the block-sparse forward, uint8 [B][H][nb][nb], nb =
    ceil(N / block), 1 = the (query block, key block) pair takes part.

    "random": each pair marked independently with probability ``density``
    (seed + 4 stream).  "local": query block i marks key blocks within
    ``window`` of i plus key block 0 (a sliding window with one global block),
    the same for every head."""
    nb = -(-N // block)
    if pattern == "random":
        g = torch.Generator(device="cpu").manual_seed(seed + 4)
        m = (torch.rand((B, H, nb, nb), generator=g) < density).to(torch.uint8)
    elif pattern == "local":
        i = torch.arange(nb)
        band = ((i[:, None] - i[None, :]).abs() <= window) | (i[None, :] == 0)
        m = band.to(torch.uint8).expand(B, H, nb, nb).clone()
    else:
        raise ValueError(pattern)
    return m.contiguous()


def make_key_mask(B: int, H: int, N: int, frac: float, seed: int = 0,
                  force_masked_heads_every: int = 4, force_masked_keys: int = 4):
    """Additive key-padding mask, float32 [B][H][N], entries 0 or -inf.

    Each (b, h, key) is masked independently with probability ``frac``
    (seed + 1 stream, so it does not disturb Q/K/V).  In heads with
    h % force_masked_heads_every == 0 the first ``force_masked_keys`` keys are
    masked too, so that under a causal mask the first rows of those heads
    have no allowed key at all (fully masked rows).
    """
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    u = torch.rand((B, H, N), generator=g, dtype=torch.float32)
    m = torch.zeros((B, H, N), dtype=torch.float32)
    m[u < frac] = float("-inf")
    if force_masked_heads_every > 0 and force_masked_keys > 0:
        for h in range(0, H, force_masked_heads_every):
            m[:, h, :min(force_masked_keys, N)] = float("-inf")
    return m.contiguous()


def make_inputs(w: Workload, seed: int = 0, N: int | None = None):
    """(q, k, v, key_mask or None) for a workload, all on the CPU."""
    n = w.N if N is None else N
    q, k, v = make_qkv(w.B, w.H, n, w.d, w.dtype, seed, w.qk_scale)
    mask = make_key_mask(w.B, w.H, n, w.mask_frac, seed) if w.mask_frac > 0 else None
    return q, k, v, mask


def sample_rows(B: int, H: int, N: int, frac: float, seed: int = 0, extra=()):
    """Seeded subset of flat row ids (bh*N + i): about ``frac`` of all rows,
    always with rows 0..3 and N-1 of every head plus any ids in ``extra``."""
    g = torch.Generator(device="cpu").manual_seed(seed + 2)
    total = B * H * N
    k = max(1, int(total * frac))
    pick = torch.randperm(total, generator=g)[:k]
    must = []
    for bh in range(B * H):
        for i in list(range(min(4, N))) + [N - 1]:
            must.append(bh * N + i)
    rows = torch.unique(torch.cat([pick, torch.tensor(must + list(extra), dtype=torch.int64)]))
    return rows.numpy()
