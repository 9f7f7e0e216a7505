"""Shared test helpers: marshalling between torch, numpy and the oracle, and
the GEMM error bound |gpu - oracle| <= 2e-3 * sum_k |a b| * s_a * s_b."""
import numpy as np
import torch

import synthetic

BOUND = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.bf16_bits(t)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def f32bits(x) -> np.ndarray:
    return np.asarray(x, np.float32).view(np.uint32)


def assert_gemm_bound(got: torch.Tensor, D: np.ndarray, Dabs: np.ndarray, prev=None, what=""):
    """Elementwise bound against the unrounded fp64 oracle.

    The bound holds for the FP32 result of the GEMM.  A bf16 output adds one
    round-to-nearest-even to bf16 (unit roundoff 2^-8), which the bound
    cannot absorb where |y| is close to sum|a b| (all products of one sign):
    there the tolerance grows by 2^-8 |y|.  With an FP32 accumulation buffer,
    `prev` (its old contents) adds one fp32 rounding of the sum."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    tol = BOUND * Dabs
    if got.dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * (np.abs(D) + BOUND * Dabs)
    if prev is not None:
        tol = tol + 2.0 ** -23 * (np.abs(np.asarray(prev, np.float64)) + np.abs(D))
    err = np.abs(g - D)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} entries outside the bound; first {idx.tolist()}: "
            f"got {g[tuple(idx.T)]}, want {D[tuple(idx.T)]}, tol {tol[tuple(idx.T)]}")
