"""Seeded synthetic inputs for the frame-wise GDN forward pass.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, imports nothing from the rest of the package, and is the
only code shared by the CUDA-path tests and the fp64 oracle tests.

Distributions (the shapes stand in for a latent video: H*D = 2240 model width in
20 heads, 880 tokens per latent frame from a 40 x 22 latent grid, up to 121
latent frames):
  q, k, v ~ N(0, 1), rounded to bf16 for the bf16 path (kept fp32 otherwise);
  beta    = sigmoid(N(0, 1))            per (batch, token, head), fp32;
  gamma   = exp(-softplus(N(0, 1)))     per (batch, frame, head), fp32;
  S_0     = 0, or N(0, s0_std^2)        per (batch, head), fp32.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass
class GdnInputs:
    q: torch.Tensor      # [B, F*N, H, D]
    k: torch.Tensor      # [B, F*N, H, D]
    v: torch.Tensor      # [B, F*N, H, D]
    beta: torch.Tensor   # [B, F*N, H] fp32
    gamma: torch.Tensor  # [B, F, H] fp32
    S0: Optional[torch.Tensor]  # [B, H, D, D] fp32 or None
    B: int
    H: int
    F: int
    N: int
    D: int


def make_inputs(B: int, H: int, F: int, N: int, D: int, *, dtype: str = "bf16",
                seed: int = 0, device="cpu", s0_std: float = 0.0) -> GdnInputs:
    """Draw one seeded input set directly on ``device`` (same seed -> same values on that device)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    shape = (B, F * N, H, D)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]

    def normal(*s):
        return torch.randn(*s, generator=g, device=dev, dtype=torch.float32)

    q = normal(*shape).to(tdt)
    k = normal(*shape).to(tdt)
    v = normal(*shape).to(tdt)
    beta = torch.sigmoid(normal(B, F * N, H))
    gamma = torch.exp(-torch.nn.functional.softplus(normal(B, F, H)))
    S0 = normal(B, H, D, D) * float(s0_std) if s0_std > 0 else None
    return GdnInputs(q, k, v, beta.contiguous(), gamma.contiguous(), S0, B, H, F, N, D)


# Named workloads: (B, H, F, N, D, dtype, s0_std).
WORKLOADS = {
    "tiny_f32": (1, 1, 4, 8, 16, "f32", 0.0),
    "single_head": (1, 1, 16, 880, 112, "bf16", 0.0),
    "layer_60s_720p": (1, 20, 121, 880, 112, "bf16", 0.0),
    "streaming_60s_720p": (1, 20, 121, 880, 112, "bf16", 0.1),
    "cfg_b2_n220": (2, 20, 121, 220, 112, "bf16", 0.0),
    "cfg_b2_n880": (2, 20, 121, 880, 112, "bf16", 0.0),
    "cfg_b2_n3520": (2, 20, 121, 3520, 112, "bf16", 0.0),
}


def make_workload(name: str, *, seed: int = 0, device="cpu", F: Optional[int] = None) -> GdnInputs:
    B, H, F0, N, D, dtype, s0 = WORKLOADS[name]
    return make_inputs(B, H, F0 if F is None else F, N, D, dtype=dtype, seed=seed,
                       device=device, s0_std=s0)


@dataclass
class BlockInputs:
    x: torch.Tensor       # [B, F*N, H*D] bf16
    W_in: torch.Tensor    # [3*H*D + 2*H, H*D] bf16
    W_out: torch.Tensor   # [H*D, H*D] bf16
    S0: Optional[torch.Tensor]
    B: int
    H: int
    F: int
    N: int
    D: int


def make_block_inputs(B: int, H: int, F: int, N: int, D: int = 112, *, seed: int = 0, device="cpu",
                      s0_std: float = 0.0) -> BlockInputs:
    """Seeded synthetic block input and random-init weights (no trained weights exist here):
    x ~ N(0, 1); W_in, W_out ~ N(0, 1 / (H*D)) (unit-variance projections), all rounded to bf16;
    S_0 = 0 or N(0, s0_std^2)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    HD = H * D

    def normal(*s):
        return torch.randn(*s, generator=g, device=dev, dtype=torch.float32)

    x = normal(B, F * N, HD).to(torch.bfloat16)
    W_in = (normal(3 * HD + 2 * H, HD) / HD ** 0.5).to(torch.bfloat16)
    W_out = (normal(HD, HD) / HD ** 0.5).to(torch.bfloat16)
    S0 = normal(B, H, D, D) * float(s0_std) if s0_std > 0 else None
    return BlockInputs(x, W_in, W_out, S0, B, H, F, N, D)
