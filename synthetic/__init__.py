"""Seeded synthetic inputs shaped like the workloads of the scaled FP8 linear.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds none of the method's arithmetic (no scaling, no
FP8 encoding): it only draws bf16 tensors with the value distributions that
"Mixed Precision LLM Training: The Complete Guide" describes for the
tensors an FP8 linear sees -- activations with rare large outliers and
outlier channels ("FP8 under the hood": activation outliers; "Numerical-
failure taxonomy"), small weights, very small gradients, and heavy-tailed
per-row magnitudes for the block-wise recipe.

Every generator takes a seed and a device; the same seed on the same device
type gives the same tensor.  The values are drawn in fp32 and rounded to
bf16 by torch's cast (round to nearest even).
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """bf16 tensor with entries ~ N(0, std^2)."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def with_outlier_entries(shape, std: float, frac: float, factor: float, seed: int,
                         device="cpu") -> torch.Tensor:
    """N(0, std^2) entries; exactly round(frac * numel) seeded positions are
    multiplied by `factor` (activation outliers)."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std
    n = x.numel()
    k = int(round(frac * n))
    if k:
        idx = torch.randperm(n, generator=g, device=device)[:k]
        x.view(-1)[idx] *= factor
    return x.to(torch.bfloat16)


def with_outlier_channels(shape, std: float, n_channels: int, factor: float, seed: int,
                          device="cpu") -> torch.Tensor:
    """N(0, std^2) entries; `n_channels` seeded columns (input features) are
    multiplied by `factor` (outlier channels)."""
    g = _gen(seed, device)
    rows, cols = shape
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * std
    if n_channels:
        ch = torch.randperm(cols, generator=g, device=device)[:n_channels]
        x[:, ch] *= factor
    return x.to(torch.bfloat16)


def _student_t(shape, nu: int, g: torch.Generator, device) -> torch.Tensor:
    """Student-t with integer `nu` degrees of freedom: Z / sqrt(chi2_nu / nu),
    chi2_nu drawn as a sum of nu squared standard normals."""
    z = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(*shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2 += torch.randn(*shape, generator=g, device=device, dtype=torch.float32) ** 2
    return z / torch.sqrt(chi2 / nu)


def student_t(shape, nu: int, scale: float, seed: int, device="cpu") -> torch.Tensor:
    """bf16 entries scale * t_nu (heavy tails: exercises saturation when the
    scale is stale and underflow when it is small)."""
    g = _gen(seed, device)
    return (_student_t(shape, nu, g, device) * scale).to(torch.bfloat16)


def student_t_rows(shape, std: float, nu: int, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) entries, each row multiplied by |t_nu| (per-row heavy-tailed
    magnitudes, the case block-wise scaling is for)."""
    g = _gen(seed, device)
    rows, cols = shape
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * std
    r = _student_t((rows, 1), nu, g, device).abs()
    return (x * r).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor's bit patterns."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)
