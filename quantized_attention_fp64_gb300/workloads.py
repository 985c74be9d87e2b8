"""Seeded synthetic inputs for the benchmark configurations.

This module holds no arithmetic of the method; it only draws the BF16 Q, K
and V tensors that both the library and the test oracle consume. Shapes and
value distributions follow the five benchmark configurations (diffusion
self-attention with 28 heads of dimension 128 at image and video sizes, plus
a long-sequence case past 100k tokens), and head dimension 64 (the pages'
second workload) at the image and video sizes. Each tensor is drawn in fp32 from a
torch generator seeded with ``1000 + index`` (per-channel key offsets use the
next seed) and rounded to bf16.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    S: int
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    k_offset_std: float = 0.0   # per-(head, channel) key offset shared over batch and tokens
    outlier_p: float = 0.0      # probability that a Q or K entry is scaled by outlier_scale
    outlier_scale: float = 8.0
    smooth_k: bool = True
    D: int = 128                # head dimension

    @property
    def attention_ops(self) -> int:
        """4 * B * H * S^2 * D: the multiply-adds of QK^T and PV, counted as 2 ops each."""
        return 4 * self.B * self.H * self.S * self.S * self.D


WORKLOADS = {
    w.name: w
    for w in [
        Workload("B1_H2_S256", 0, 1, 2, 256, smooth_k=False),
        Workload("B2_H8_S1024", 1, 2, 8, 1024, k_offset_std=3.0),
        Workload("B1_H28_S4096", 2, 1, 28, 4096, k_offset_std=2.0),
        Workload("B1_H28_S16384", 3, 1, 28, 16384, q_std=1.5, k_std=1.5, outlier_p=0.01),
        Workload("B1_H28_S131072", 4, 1, 28, 131072, k_offset_std=2.0),
        Workload("B1_H80_S131072", 5, 1, 80, 131072, k_offset_std=2.0),
        Workload("B1_H28_S4096_D64", 6, 1, 28, 4096, k_offset_std=2.0, D=64),
        Workload("B1_H28_S16384_D64", 7, 1, 28, 16384, q_std=1.5, k_std=1.5, outlier_p=0.01, D=64),
    ]
}


def custom(B: int, H: int, S: int, seed_index: int = 100, **kw) -> Workload:
    return Workload(f"B{B}_H{H}_S{S}", seed_index, B, H, S, **kw)


def make_qkv(w: Workload, device="cuda", layout: str = "NHD"):
    """Draws (q, k, v) as BF16 tensors of shape [B,S,H,D] ("NHD") or
    [B,H,S,D] ("HND"), contiguous, on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + w.index)
    shape = (w.B, w.S, w.H, w.D)

    def draw(std, outliers):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if outliers and w.outlier_p > 0:
            mask = torch.rand(shape, generator=gen, device=device) < w.outlier_p
            x = torch.where(mask, x * w.outlier_scale, x)
        return x.to(torch.bfloat16)

    q = draw(w.q_std, True)
    k32 = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if w.k_std != 1.0:
        k32.mul_(w.k_std)
    if w.outlier_p > 0:
        mask = torch.rand(shape, generator=gen, device=device) < w.outlier_p
        k32 = torch.where(mask, k32 * w.outlier_scale, k32)
    if w.k_offset_std > 0:
        g2 = torch.Generator(device=device)
        g2.manual_seed(1000 + w.index + 1)
        off = torch.randn((w.H, w.D), generator=g2, device=device, dtype=torch.float32) * w.k_offset_std
        k32.add_(off[None, None])
    k = k32.to(torch.bfloat16)
    del k32
    v = draw(w.v_std, False)
    if layout == "HND":
        q, k, v = (t.transpose(1, 2).contiguous() for t in (q, k, v))
    elif layout != "NHD":
        raise ValueError(layout)
    return q, k, v
