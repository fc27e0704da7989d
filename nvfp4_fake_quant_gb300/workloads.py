"""Seeded synthetic inputs shared by the tests, ``bench.py`` and the CPU oracle.

Only input generation lives here: no step of the quantizer or of attention.
Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
as fp32 and rounded to bf16 (RNE), so the GPU path and the oracle see the same
bytes.  Layout of attention tensors: [B, N, H, D] contiguous.

Workloads (shapes of the Wan2.1-T2V-1.3B attention that the "Attn-QAT
Training" guide trains; 12 heads of 128 from the "vsqa-preview-1.3b
metadata.json" architecture, latent grids from its training geometry):
  tiny        B=1, H=2, N=256, D=64, q/k/v/dO iid N(0,1), seed 0, scale 1/8
  vsa25088    B=1, H=12, N=25088 (16x28x56 latent), D=128, q/k/v/dO iid N(0,1),
              seed 4 (block-sparse: 196 cubes of 4x4x8, top-20 key cubes each)
  quant       X bf16 [4096, 4096] N(0,1); 1% of entries (uniform, without
              replacement) multiplied by 50; then 2% of the 16-element blocks
              zeroed; seed 1
  wan25088    B=1, H=12, D=128, N=25088 (16x28x56 latent tokens); Q, K N(0,1)
              with every (token, head) row scaled to unit RMS over D; V, dO
              N(0,1); seed 2
  wan_ffn_up  the NVFP4 linear on the Wan FFN up-projection: x [25088, 1536]
              (the 16x28x56 latent tokens, hidden 12 x 128) N(0,1), w [8960, 1536]
              N(0, 1/1536), bias [8960] N(0, 0.01), grad [25088, 8960] N(0,1);
              seed 6 (ffn_dim 8960 from the metadata's architecture)
  wan32760    B=1, H=12, D=128, N=32760 (21x30x52); Q, K N(0,1) times a
              per-(head, channel) factor exp(N(0,1)) (one set for Q, one for
              K); V, dO N(0,1); seed 3
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BF16 = torch.bfloat16


@dataclass
class AttnInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    scale: float
    causal: bool = False

    @property
    def shape(self):
        b, nq, h, d = self.q.shape
        return b, nq, self.k.shape[1], h, d


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _randn(g, *shape) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def attn_inputs(b, nq, nkv, h, d, seed, scale=None, causal=False, dist="normal") -> AttnInputs:
    """Generic attention inputs: iid N(0,1) q, k, v, dO (``dist="normal"``),
    or q/k rows scaled to unit RMS over D (``dist="unit_rms"``), or q/k with
    per-(head, channel) lognormal(0,1) factors (``dist="lognormal_channels"``).
    """
    g = _gen(seed)
    q = _randn(g, b, nq, h, d)
    k = _randn(g, b, nkv, h, d)
    v = _randn(g, b, nkv, h, d)
    do = _randn(g, b, nq, h, d)
    if dist == "unit_rms":
        q = q / q.pow(2).mean(dim=-1, keepdim=True).sqrt()
        k = k / k.pow(2).mean(dim=-1, keepdim=True).sqrt()
    elif dist == "lognormal_channels":
        cq = torch.exp(_randn(g, h, d))
        ck = torch.exp(_randn(g, h, d))
        q = q * cq
        k = k * ck
    elif dist != "normal":
        raise ValueError(dist)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    return AttnInputs(q.to(BF16), k.to(BF16), v.to(BF16), do.to(BF16), scale, causal)


def tiny() -> AttnInputs:
    return attn_inputs(1, 256, 256, 2, 64, seed=0, scale=1.0 / 8.0)


def wan25088() -> AttnInputs:
    return attn_inputs(1, 25088, 25088, 12, 128, seed=2, dist="unit_rms")


def wan32760() -> AttnInputs:
    return attn_inputs(1, 32760, 32760, 12, 128, seed=3, dist="lognormal_channels")


# Latent grid of the block-sparse workload (Wan2.1-1.3B at 448x896x61 frames:
# 16 x 28 x 56 tokens) and its cube shape (4 x 4 x 8 = 128 tokens per cube).
VSA_GRID = (16, 28, 56)
VSA_CUBE = (4, 4, 8)


def vsa25088() -> AttnInputs:
    """Block-sparse workload: B=1, H=12, N=25088, D=128, q/k/v/dO iid N(0,1), seed 4,
    tokens in raster (t, h, w) order of the VSA_GRID latent."""
    return attn_inputs(1, 25088, 25088, 12, 128, seed=4)


def quant_matrix(rows=4096, cols=4096, seed=1, outlier_frac=0.01, outlier_mul=50.0,
                 zero_block_frac=0.02) -> torch.Tensor:
    """The standalone-quantizer matrix (bf16 [rows, cols], cols % 16 == 0)."""
    assert cols % 16 == 0
    g = _gen(seed)
    x = _randn(g, rows, cols)
    flat = x.view(-1)
    n_out = int(round(outlier_frac * flat.numel()))
    idx = torch.randperm(flat.numel(), generator=g)[:n_out]
    flat[idx] *= outlier_mul
    blocks = x.view(-1, 16)
    n_zero = int(round(zero_block_frac * blocks.shape[0]))
    bidx = torch.randperm(blocks.shape[0], generator=g)[:n_zero]
    blocks[bidx] = 0.0
    return x.to(BF16)


def random_matrix(rows, cols, seed, scale=1.0) -> torch.Tensor:
    """Plain N(0, scale^2) bf16 matrix (parity cases of other sizes)."""
    return (_randn(_gen(seed), rows, cols) * scale).to(BF16)


WAN_HIDDEN, WAN_FFN = 1536, 8960


@dataclass
class LinearInputs:
    x: torch.Tensor      # bf16 [M, K]
    w: torch.Tensor      # bf16 [N, K]
    bias: torch.Tensor   # bf16 [N]
    grad: torch.Tensor   # bf16 [M, N]


def linear_inputs(m, n, k, seed) -> LinearInputs:
    g = _gen(seed)
    x = _randn(g, m, k).to(BF16)
    w = (_randn(g, n, k) * k ** -0.5).to(BF16)
    bias = (_randn(g, n) * 0.1).to(BF16)
    grad = _randn(g, m, n).to(BF16)
    return LinearInputs(x, w, bias, grad)


def wan_ffn_up() -> LinearInputs:
    return linear_inputs(25088, WAN_FFN, WAN_HIDDEN, seed=6)
