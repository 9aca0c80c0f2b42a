"""Seeded synthetic inputs for the Direct-P attention forward.

This module holds the workload shapes and the random draws only -- none of the
method's arithmetic -- so that the CUDA path and the CPU oracle can be fed the
same bytes.  All draws use a CPU ``torch.Generator`` in fp32 and are cast to
bf16 at the end.  The pages measure on model workloads (a 14B video DiT,
Llama-style LLMs); these tensors stand in for them with the shapes and value
structure of the five workload definitions below.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    index: int
    B: int
    H: int
    N: int
    D: int
    recipe: str
    description: str

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.D)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> int:
        """Attention FLOPs counted as 4*B*H*N^2*D (two N x N x D products)."""
        return 4 * self.B * self.H * self.N * self.N * self.D

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def name(self) -> str:
        return "B%d_H%d_N%d_D%d_%s" % (self.B, self.H, self.N, self.D, self.recipe)


WORKLOADS = {
    1: Workload(1, 1, 1, 256, 64, "normal", "Q,K,V ~N(0,1)"),
    2: Workload(2, 1, 8, 4096, 128, "outlier_channels",
                "Q,K,V ~N(0,1); per tensor and head, 4 random channels scaled x8"),
    3: Workload(3, 2, 16, 8192, 128, "channel_std",
                "Q,K per-(head, channel) std log-uniform in [0.25, 4]; V ~N(0,1)"),
    4: Workload(4, 1, 40, 32768, 128, "token_rms",
                "video-DiT shape; Q,K rows scaled by r~U[0.5,2] per token; V ~N(0,1)"),
    5: Workload(5, 4, 16, 16384, 64, "spiky_tokens",
                "Q,K,V ~N(0,1); 2% of token indices per batch element scaled x6"),
}


def _randn(g, shape):
    return torch.randn(shape, generator=g, dtype=torch.float32)


def make_inputs(w: Workload, seed: int | None = None):
    """Returns (q, k, v) as contiguous CPU bf16 tensors of shape [B,H,N,D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape = w.shape
    B, H, N, D = shape
    q = _randn(g, shape)
    k = _randn(g, shape)
    v = _randn(g, shape)
    if w.recipe == "normal":
        pass
    elif w.recipe == "outlier_channels":
        for t in (q, k, v):
            for b in range(B):
                for h in range(H):
                    ch = torch.randperm(D, generator=g)[:4]
                    t[b, h, :, ch] *= 8.0
    elif w.recipe == "channel_std":
        lo, hi = math.log(0.25), math.log(4.0)
        for t in (q, k):
            u = torch.rand((1, H, 1, D), generator=g, dtype=torch.float32)
            t *= torch.exp(lo + (hi - lo) * u)
    elif w.recipe == "token_rms":
        for t in (q, k):
            r = 0.5 + 1.5 * torch.rand((B, H, N, 1), generator=g, dtype=torch.float32)
            t *= r
    elif w.recipe == "spiky_tokens":
        nspike = max(1, int(round(0.02 * N)))
        for b in range(B):
            idx = torch.randperm(N, generator=g)[:nspike]
            for t in (q, k, v):
                t[b, :, idx, :] *= 6.0
    else:
        raise ValueError("unknown recipe %r" % w.recipe)
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v))


def make_custom(B, H, N, D, seed, kind="normal", scale=1.0):
    """Small ad-hoc inputs for edge-case tests (ragged N, zeros, constants)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, D)
    if kind == "normal":
        ts = [_randn(g, shape) * scale for _ in range(3)]
    elif kind == "zeros":
        ts = [torch.zeros(shape) for _ in range(3)]
    elif kind == "zero_q":
        ts = [torch.zeros(shape), _randn(g, shape) * scale, _randn(g, shape) * scale]
    elif kind == "wide":
        # log-uniform magnitudes over many binades, random signs
        ts = []
        for _ in range(3):
            mag = torch.exp(torch.empty(shape).uniform_(-20.0, 12.0, generator=g))
            sgn = torch.where(torch.rand(shape, generator=g) < 0.5, -1.0, 1.0)
            ts.append(mag * sgn)
    else:
        raise ValueError(kind)
    return tuple(t.to(torch.bfloat16).contiguous() for t in ts)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
