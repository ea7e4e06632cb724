"""Seeded synthetic inputs for the SANA-Video linear-attention layer.

This module only *makes inputs*; it holds none of the attention arithmetic.
Both the CUDA path and the FP64 oracle are fed from it, so every parity test
compares the two on the very same tensors.

What it stands in for: the activations that reach the linear-attention core
of ``SanaVideoLinearAttention.forward`` on the page "PR #35728 完整报告 -
[diffusion] Accelerate SANA-Video linear attention in quality=high"
(section 关键源码片段, snippet ``sana_video.py``): per-head RMSNorm'd Q and K
pass through ReLU, are rotated by an interleaved RoPE (only the rotated copies
feed the two GEMMs), and the un-rotated ReLU'd Q and K give the normalizer.
The RMSNorm/projection weights are not available, so standard normals stand in
for their output.

Recipe (draw order is fixed; one ``torch.Generator`` seeded with ``seed``):
  1. ``q_pre = relu(randn)``, ``k_pre = relu(randn)`` -> BF16
  2. ``v = randn`` -> BF16
  3. ``q_rot``/``k_rot`` = interleaved RoPE of ``q_pre``/``k_pre`` (FP32 maths
     on the BF16 values) -> BF16.  Pair ``(2p, 2p+1)`` of an axis chunk of
     width ``d`` is turned by ``pos * 10000**(-2p/d)``.  With a latent grid
     ``(T, Hg, W)`` the head dim is cut into (t, h, w) chunks of widths
     ``(D - 4*(D//6), 2*(D//6), 2*(D//6))`` and tokens run t-major, then h,
     then w; without a grid one chunk of width D uses ``pos = token index``.
  4. ``den[h, n] = q_pre[h, n, :] . sum_m k_pre[h, m, :] + 1e-6`` in FP64,
     rounded once to FP32 (a denominator: the layer divides by it).

All tensors are contiguous ``[1, H, N, D]`` (``den``: ``[1, H, N, 1]``).  On request the
generator also returns the pre-ReLU ``q``, ``k`` and the FP32 rotation tables, the inputs
of the fused producer path.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

EPS = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    heads: int
    tokens: int
    head_dim: int
    grid: tuple[int, int, int] | None  # latent (frames, height, width) or None for 1-D positions
    seed: int = 0


# Shapes of the two SANA-Video profiles the pages time (832x480, 81 frames and
# 1280x736, 193 frames, T2V) at the VAE/patch stride that gives the latent
# grids below, plus the small case used for brute-force checks.
WORKLOADS = {
    "tiny": Workload("tiny", 2, 256, 32, None),
    "480p_81f": Workload("480p_81f", 20, 32760, 112, (21, 30, 52)),
    "720p_193f": Workload("720p_193f", 20, 180320, 112, (49, 46, 80)),
    "720p_193f_d64": Workload("720p_193f_d64", 32, 180320, 64, (49, 46, 80)),
}
# Token-count sweep at the 720p head shape (powers of two, 1-D positions).
SWEEP_TOKENS = tuple(1 << k for k in range(12, 19))  # 4096 .. 262144
for _n in SWEEP_TOKENS:
    WORKLOADS[f"sweep_n{_n}"] = Workload(f"sweep_n{_n}", 20, _n, 112, None)
    WORKLOADS[f"sweep_n{_n}_d64"] = Workload(f"sweep_n{_n}_d64", 32, _n, 64, None)
# A denoise step touches this many linear-attention layers, each with its own inputs.
DENOISE_LAYERS = 20


def _axis_chunks(head_dim: int, grid) -> list[tuple[int, int]]:
    """(start, width) of each RoPE axis chunk inside the head dim."""
    if grid is None:
        return [(0, head_dim)]
    third = 2 * (head_dim // 6)
    wt = head_dim - 2 * third
    return [(0, wt), (wt, third), (wt + third, third)]


def _positions(tokens: int, grid, device) -> list[torch.Tensor]:
    n = torch.arange(tokens, device=device, dtype=torch.int64)
    if grid is None:
        return [n]
    t, hg, w = grid
    if t * hg * w != tokens:
        raise ValueError(f"grid {grid} does not hold {tokens} tokens")
    return [n // (hg * w), (n // w) % hg, n % w]


def rope_tables(tokens: int, head_dim: int, grid=None, device="cpu"):
    """cos/sin of the rotation angle for every (token, pair): FP32 [N, D/2]."""
    pos = _positions(tokens, grid, device)
    cos = torch.empty(tokens, head_dim // 2, dtype=torch.float32, device=device)
    sin = torch.empty_like(cos)
    for (start, width), p in zip(_axis_chunks(head_dim, grid), pos):
        if width == 0:
            continue
        pair = torch.arange(width // 2, device=device, dtype=torch.float64)
        freq = torch.pow(torch.tensor(10000.0, dtype=torch.float64, device=device), -2.0 * pair / width)
        ang = p.to(torch.float64)[:, None] * freq[None, :]
        cos[:, start // 2:(start + width) // 2] = torch.cos(ang).to(torch.float32)
        sin[:, start // 2:(start + width) // 2] = torch.sin(ang).to(torch.float32)
    return cos, sin


def _rotate_pairs(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor) -> torch.Tensor:
    """Interleaved rotation of (x[2p], x[2p+1]) pairs; x is FP32 [H, N, D]."""
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = x0 * cos - x1 * sin
    out[..., 1::2] = x0 * sin + x1 * cos
    return out


def make_layer(heads: int, tokens: int, head_dim: int, seed: int = 0, grid=None, device="cpu",
               producer_inputs: bool = False):
    """One layer's inputs: dict of q_rot, k_rot, v (BF16) and den (FP32).

    With producer_inputs, also the tensors the layer starts from before ReLU, RoPE and the
    normaliser: "q", "k" (BF16 [1, H, N, D], the normalised projections before ReLU) and
    the rotation tables "rope_cos", "rope_sin" (FP32 [N, D/2])."""
    if head_dim % 2:
        raise ValueError("head_dim must be even for pairwise RoPE")
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (heads, tokens, head_dim)
    q_in = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    k_in = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    q_pre, k_pre = torch.relu(q_in), torch.relu(k_in)
    v = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    cos, sin = rope_tables(tokens, head_dim, grid, device)
    q_rot = _rotate_pairs(q_pre.float(), cos, sin).to(torch.bfloat16)
    k_rot = _rotate_pairs(k_pre.float(), cos, sin).to(torch.bfloat16)
    ksum = k_pre.double().sum(dim=1)  # [H, D]
    den = (torch.einsum("hnd,hd->hn", q_pre.double(), ksum) + EPS).to(torch.float32)
    del q_pre, k_pre, ksum
    out = {
        "q_rot": q_rot.unsqueeze(0).contiguous(),
        "k_rot": k_rot.unsqueeze(0).contiguous(),
        "v": v.unsqueeze(0).contiguous(),
        "den": den.reshape(1, heads, tokens, 1).contiguous(),
    }
    if producer_inputs:
        out.update(q=q_in.unsqueeze(0).contiguous(), k=k_in.unsqueeze(0).contiguous(),
                   rope_cos=cos.contiguous(), rope_sin=sin.contiguous())
    return out


def make_anchor_layer(heads: int, tokens: int, head_dim: int, seed: int = 0, logit_scale: float = 1.0,
                      device="cpu"):
    """Inputs of a softmax anchor layer: q, k, v BF16 [1, H, N, D] ~ N(0, 1), q scaled by
    `logit_scale` (spreads the attention logits)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (1, heads, tokens, head_dim)
    q = (torch.randn(shape, generator=g, device=device) * logit_scale).to(torch.bfloat16)
    k = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    v = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v}


def make_workload(w: Workload, device="cpu", producer_inputs: bool = False):
    return make_layer(w.heads, w.tokens, w.head_dim, w.seed, w.grid, device, producer_inputs)
