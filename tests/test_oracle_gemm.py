"""Pins of the oracle's scaled FP8 GEMM and linear composition.

Sources: "Mixed Precision LLM Training: The Complete Guide", sections
"Transformer Engine internals" > "Per-tensor scaling" (the matmul result is
multiplied by the inverse scales), "Skipping the BAcc accumulator
promotion" and "DeepSeek FP8 training recipe" > "Mixed-precision
accumulation" (wide accumulation), "Block-wise scaling at 128 granularity"
(scales applied inside the matmul), "The HYBRID recipe" (E4M3 forward,
E5M2 gradients), "FP8 and gradient accumulation" (FP32 wgrad buffer).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2, GRAN_1x128, GRAN_128x128, GRAN_TENSOR

TORCH_FMT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _torch_decode(codes, fmt):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(TORCH_FMT[fmt]).to(
        torch.float64).numpy()


def _int_codes(rng, shape, fmt, lo=-8, hi=8):
    """Codes of small integers (exact in both formats for |v| <= 8)."""
    vals = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return oracle.encode(vals, fmt), vals.astype(np.int64)


@pytest.mark.parametrize("M,N,K", [(16, 32, 128), (32, 16, 32), (128, 128, 16), (5, 7, 48)])
@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_brute_force_integer_gemm(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 1000 + N + K)
    A, ai = _int_codes(rng, (M, K), fa)
    B, bi = _int_codes(rng, (N, K), fb)
    sa, sb = np.float32(0.25), np.float32(3.0)
    D, Dabs = oracle.gemm(A, fa, B, fb, sa, sb)
    exact = (ai @ bi.T).astype(np.float64) * 0.75
    assert np.array_equal(D, exact)
    assert np.array_equal(Dabs, (np.abs(ai) @ np.abs(bi).T).astype(np.float64) * 0.75)


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3), (E4M3, E5M2)])
def test_random_codes_against_library_matmul(fa, fb):
    # every finite code, decoded by torch and multiplied by numpy in fp64
    rng = np.random.default_rng(1)
    M, N, K = 33, 47, 256

    def finite_codes(fmt, shape):
        c = rng.integers(0, 256, size=shape).astype(np.uint8)
        bad = ~np.isfinite(_torch_decode(c, fmt))
        c[bad] = 0x38 if fmt == E4M3 else 0x3C
        return c

    A, B = finite_codes(fa, (M, K)), finite_codes(fb, (N, K))
    sa, sb = np.float32(1 / 448), np.float32(7.5)
    D, Dabs = oracle.gemm(A, fa, B, fb, sa, sb)
    da, db = _torch_decode(A, fa), _torch_decode(B, fb)
    ref = (da @ db.T) * (float(sa) * float(sb))
    np.testing.assert_allclose(D, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(Dabs, np.abs(da) @ np.abs(db).T * float(sa) * float(sb),
                               rtol=1e-12)
    # operand symmetry: (A B^T)^T = B A^T
    Dt, _ = oracle.gemm(B, fb, A, fa, sb, sa)
    np.testing.assert_allclose(Dt, D.T, rtol=1e-12, atol=1e-300)


def test_all_ones():
    K = 640
    one = oracle.encode(np.ones(1, np.float32), E4M3)[0]
    A = np.full((16, K), one, np.uint8)
    B = np.full((32, K), one, np.uint8)
    D, _ = oracle.gemm(A, E4M3, B, E4M3, np.float32(0.5), np.float32(0.125))
    assert (D == K * 0.0625).all()


def test_sampled_entries_equal_full_gemm():
    rng = np.random.default_rng(4)
    A = rng.integers(0, 0x7E, size=(64, 256)).astype(np.uint8)
    B = rng.integers(0, 0x7E, size=(48, 256)).astype(np.uint8)
    D, Dabs = oracle.gemm(A, E4M3, B, E4M3, 0.5, 2.0)
    ii = rng.integers(0, 64, 100)
    jj = rng.integers(0, 48, 100)
    d, dabs = oracle.gemm_entries(A, E4M3, B, E4M3, 0.5, 2.0, ii, jj)
    assert np.array_equal(d, D[ii, jj]) and np.array_equal(dabs, Dabs[ii, jj])


def test_uniform_block_scales_equal_per_tensor():
    rng = np.random.default_rng(6)
    M, N, K = 160, 256, 384
    A, ai = _int_codes(rng, (M, K), E4M3)
    B, bi = _int_codes(rng, (N, K), E4M3)
    sa = np.full((M, K // 128), 0.5, np.float32)
    sb = np.full((N // 128, K // 128), 4.0, np.float32)
    Db, _ = oracle.gemm(A, E4M3, B, E4M3, sa, sb, GRAN_1x128, GRAN_128x128)
    Dt, _ = oracle.gemm(A, E4M3, B, E4M3, 0.5, 4.0)
    assert np.array_equal(Db, Dt)
    assert np.array_equal(Dt, (ai @ bi.T).astype(np.float64) * 2.0)


@pytest.mark.parametrize("ga,gb", [(GRAN_1x128, GRAN_128x128), (GRAN_128x128, GRAN_128x128),
                                   (GRAN_1x128, GRAN_1x128), (GRAN_TENSOR, GRAN_128x128)])
def test_block_scales_against_blockwise_numpy(ga, gb):
    # independent route: decode with torch, split K into 128-blocks, weight
    # each block's partial product by the outer product of its factors
    rng = np.random.default_rng(8)
    M, N, K = 256, 256, 512
    KB = K // 128
    A, ai = _int_codes(rng, (M, K), E4M3)
    B, bi = _int_codes(rng, (N, K), E5M2)

    def scales(gran, rows):
        if gran == GRAN_TENSOR:
            return np.float32(0.75), np.full((rows, KB), 0.75)
        r = rows if gran == GRAN_1x128 else rows // 128
        s = (2.0 ** rng.integers(-6, 6, size=(r, KB))).astype(np.float32)
        full = s if gran == GRAN_1x128 else np.repeat(s, 128, axis=0)
        return s, full.astype(np.float64)

    sa, fa_full = scales(ga, M)
    sb, fb_full = scales(gb, N)
    D, _ = oracle.gemm(A, E4M3, B, E5M2, sa, sb, ga, gb)
    parts = np.einsum("mbk,nbk->mnb", ai.reshape(M, KB, 128).astype(np.float64),
                      bi.reshape(N, KB, 128).astype(np.float64))
    ref = np.einsum("mnb,mb,nb->mn", parts, fa_full, fb_full)
    assert np.array_equal(D, ref)


def test_single_nonzero_block_scale_isolates_indexing():
    rng = np.random.default_rng(10)
    M, N, K = 256, 384, 384
    A, ai = _int_codes(rng, (M, K), E4M3)
    B, bi = _int_codes(rng, (N, K), E4M3)
    sa = np.zeros((M, 3), np.float32)
    sb = np.zeros((3, 3), np.float32)
    sa[77, 2] = 2.0
    sb[1, 2] = 8.0
    D, _ = oracle.gemm(A, E4M3, B, E4M3, sa, sb, GRAN_1x128, GRAN_128x128)
    nz = np.argwhere(D != 0)
    assert set(map(int, nz[:, 0])) <= {77}
    assert set(map(int, nz[:, 1])) <= set(range(128, 256))
    want = (ai[77, 256:] @ bi[128:256, 256:].T) * 16.0
    assert np.array_equal(D[77, 128:256], want.astype(np.float64))


def _bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_linear_fwd_with_identity_input_returns_weight():
    # X = I (M = K): Y = X W^T = W^T, dequantised
    rng = np.random.default_rng(12)
    K, N = 128, 64
    X = _bits(np.eye(K))
    W = _bits(rng.standard_normal((N, K)) * 0.02)
    rec = oracle.Recipe(scaling=oracle.SCALING_DYNAMIC)
    st = oracle.LinearState(rec)
    Y, _ = oracle.linear_fwd(X, W, rec, st)
    sw = np.float32(448) / oracle.amax(W)
    wq, _ = oracle.quantize(W, E4M3, sw)
    want = oracle.decode(wq, E4M3).T * 448.0 * float(np.float32(1) / sw) * float(np.float32(1) / np.float32(448))
    np.testing.assert_allclose(Y, want, rtol=1e-15)


def test_linear_dgrad_with_identity_weight_returns_dequantised_gradient():
    rng = np.random.default_rng(13)
    M, K = 64, 128
    rec = oracle.Recipe(scaling=oracle.SCALING_DELAYED)
    st = oracle.LinearState(rec)
    X = _bits(rng.standard_normal((M, K)))
    W = _bits(np.eye(K))
    dY = _bits(rng.standard_normal((M, K)) * 1e-3)
    oracle.linear_fwd(X, W, rec, st)
    (dX, _), _ = oracle.linear_bwd(dY, rec, st)
    # first step of delayed scaling: every scale is still 1
    dyq, _ = oracle.quantize(dY, E5M2, 1.0)
    assert np.array_equal(dX, oracle.decode(dyq, E5M2))


def test_linear_wgrad_accumulates_and_matches_definition():
    rng = np.random.default_rng(14)
    M, N, K = 96, 64, 128
    rec = oracle.Recipe(scaling=oracle.SCALING_DYNAMIC)
    st = oracle.LinearState(rec)
    X = _bits(rng.standard_normal((M, K)))
    W = _bits(rng.standard_normal((N, K)) * 0.02)
    dY = _bits(rng.standard_normal((M, N)) * 1e-3)
    oracle.linear_fwd(X, W, rec, st)
    prev = rng.standard_normal((N, K)).astype(np.float32)
    (dX, _), (dW, _) = oracle.linear_bwd(dY, rec, st, dW_prev=prev)
    sx = np.float32(448) / oracle.amax(X)
    sw = np.float32(448) / oracle.amax(W)
    sdy = np.float32(57344) / oracle.amax(dY)
    xd = oracle.decode(oracle.quantize(X, E4M3, sx)[0], E4M3) * float(np.float32(1) / sx)
    wd = oracle.decode(oracle.quantize(W, E4M3, sw)[0], E4M3) * float(np.float32(1) / sw)
    dyd = oracle.decode(oracle.quantize(dY, E5M2, sdy)[0], E5M2) * float(np.float32(1) / sdy)
    np.testing.assert_allclose(dX, dyd @ wd, rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(dW, prev + dyd.T @ xd, rtol=1e-12, atol=1e-12)


def test_delayed_linear_uses_previous_step_scale():
    # step 0 quantises with scale 1; step 1 with 448 / amax(step 0)
    rng = np.random.default_rng(15)
    rec = oracle.Recipe(scaling=oracle.SCALING_DELAYED, history_len=16)
    st = oracle.LinearState(rec)
    X0 = _bits(rng.standard_normal((32, 128)) * 2)
    X1 = _bits(rng.standard_normal((32, 128)) * 3)
    W = _bits(rng.standard_normal((16, 128)) * 0.02)
    oracle.linear_fwd(X0, W, rec, st)
    assert np.array_equal(st.x_q, oracle.quantize(X0, E4M3, 1.0)[0])
    oracle.linear_fwd(X1, W, rec, st)
    s1 = np.float32(448) / oracle.amax(X0)
    assert np.array_equal(st.x_q, oracle.quantize(X1, E4M3, s1)[0])
    assert st.roles[0].scale[0] == np.float32(448) / max(oracle.amax(X0), oracle.amax(X1))


def _dequant_blocks(q, fmt, s, block_rows):
    """Block-dequantised operand: codes times the scale of their block."""
    d = oracle.decode(q, fmt)
    f = np.repeat(np.repeat(np.asarray(s, np.float64), 128, axis=1), block_rows, axis=0)
    return d * f


def test_block_backward_against_dequantised_matmul():
    # independent route: dequantise every operand block by block, then one
    # fp64 matmul; sum_kb (sa sb) sum_k a b == sum_k (a sa)(b sb)
    rng = np.random.default_rng(21)
    M, N, K = 256, 384, 256
    rec = oracle.Recipe(scaling=oracle.SCALING_BLOCK)
    st = oracle.LinearState(rec)
    X = _bits(rng.standard_normal((M, K)) * np.abs(rng.standard_t(3, (M, 1))))
    W = _bits(rng.standard_normal((N, K)) * 0.02)
    dY = _bits(rng.standard_normal((M, N)) * 1e-3)
    oracle.linear_fwd(X, W, rec, st)
    (dX, _), (dW, _) = oracle.linear_bwd(dY, rec, st)
    dy = _dequant_blocks(*oracle.block_quantize(dY, E5M2, 1)[:1], E5M2,
                         oracle.block_quantize(dY, E5M2, 1)[1], 1)
    wq, ws = oracle.block_quantize(W, E4M3, 128)
    w = _dequant_blocks(wq, E4M3, ws, 128)
    np.testing.assert_allclose(dX, dy @ w, rtol=1e-10, atol=1e-14)
    # wgrad operands: 1x128 blocks along the tokens, i.e. of dY^T and X^T
    dytq, dyts = oracle.block_quantize(np.ascontiguousarray(dY.T), E5M2, 1)
    xtq, xts = oracle.block_quantize(np.ascontiguousarray(X.T), E4M3, 1)
    np.testing.assert_allclose(dW, _dequant_blocks(dytq, E5M2, dyts, 1)
                               @ _dequant_blocks(xtq, E4M3, xts, 1).T, rtol=1e-10, atol=1e-14)
    # the transposed weight operand is the transposed cast
    assert np.array_equal(st.wt_q, wq.T) and np.array_equal(st.wt_sinv, ws.T)


def test_row_scales_are_an_outer_product():
    rng = np.random.default_rng(41)
    M, N, K = 33, 47, 160
    A, ai = _int_codes(rng, (M, K), E4M3)
    B, bi = _int_codes(rng, (N, K), E5M2)
    sa = (2.0 ** rng.integers(-4, 4, M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-4, 4, N)).astype(np.float32)
    D, _ = oracle.gemm(A, E4M3, B, E5M2, sa, sb, oracle.GRAN_ROW, oracle.GRAN_ROW)
    want = (ai @ bi.T).astype(np.float64) * np.outer(sa, sb)
    assert np.array_equal(D, want)
    D2, _ = oracle.gemm(A, E4M3, B, E5M2, sa, np.float32(0.5), oracle.GRAN_ROW, GRAN_TENSOR)
    assert np.array_equal(D2, (ai @ bi.T).astype(np.float64) * sa[:, None] * 0.5)


def test_row_scaled_linear_against_dequantised_matmul():
    rng = np.random.default_rng(42)
    M, N, K = 64, 48, 96
    rec = oracle.Recipe(scaling=oracle.SCALING_ROW)
    st = oracle.LinearState(rec)
    X = _bits(rng.standard_normal((M, K)) * np.abs(rng.standard_t(3, (M, 1))))
    W = _bits(rng.standard_normal((N, K)) * 0.02)
    dY = _bits(rng.standard_normal((M, N)) * 1e-3)
    Y, _ = oracle.linear_fwd(X, W, rec, st)
    (dX, _), (dW, _) = oracle.linear_bwd(dY, rec, st)

    def deq(bits, fmt, axis):
        # cast with one scale per row (axis 1) or per column (axis 0), dequantised
        src = bits if axis == 1 else np.ascontiguousarray(bits.T)
        q, s = oracle.row_quantize(src, fmt)
        d = oracle.decode(q, fmt) * s[:, None].astype(np.float64)
        return d if axis == 1 else d.T

    np.testing.assert_allclose(Y, deq(X, E4M3, 1) @ deq(W, E4M3, 1).T, rtol=1e-12)
    np.testing.assert_allclose(dX, deq(dY, E5M2, 1) @ deq(W, E4M3, 0), rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(dW, deq(dY, E5M2, 0).T @ deq(X, E4M3, 0), rtol=1e-12, atol=1e-18)
