"""Pins of the oracle's scale update (delayed / history / dynamic, margin,
power-of-two) and block quantiser.

Sources: "Mixed Precision LLM Training: The Complete Guide", sections
"Transformer Engine internals" > "Per-tensor scaling", "Delayed scaling",
"History-based scaling"; "Calibration deep dive" > "Dynamic calibration";
"torch.compile and FP8" (all-zero tensors skip the update); "DeepSeek FP8
training recipe" > "Block-wise scaling at 128 granularity".  "Training and
inference of large language models using 8-bit floating point" (per-tensor
scaling bias: power-of-two scales).
"""
import os

import numpy as np
import pytest

import oracle
from oracle import ALGO_MAX, ALGO_MOST_RECENT, E4M3, E5M2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLT_MAX = np.finfo(np.float32).max
FLT_MIN = np.finfo(np.float32).tiny


def _ring_rows():
    rows = []
    for line in open(os.path.join(GOLDEN, "delayed_scaling_ring.txt")):
        if line.startswith("#") or not line.strip():
            continue
        rows.append([float(v) for v in line.split()])
    return rows


@pytest.mark.parametrize("col,algo,margin,pow2", [
    (2, ALGO_MAX, 0, False), (3, ALGO_MAX, 0, True), (4, ALGO_MAX, 1, False),
    (5, ALGO_MOST_RECENT, 0, False)])
def test_delayed_scaling_ring_golden(col, algo, margin, pow2):
    st = oracle.ScaleState(16)
    for row in _ring_rows():
        oracle.update_scale(st, row[1], algo, E4M3, margin, pow2)
        assert st.scale[0] == np.float32(row[col]), row
        assert st.scale_inv[0] == np.float32(1.0) / np.float32(row[col])
        assert st.pos[0] == (int(row[0]) + 1) % 16


def test_most_recent_equals_history_of_one():
    rng = np.random.default_rng(3)
    a = oracle.ScaleState(16)
    b = oracle.ScaleState(1)
    for t in range(40):
        amax = np.float32(abs(rng.standard_normal()) * 10.0 ** rng.integers(-3, 3))
        if t % 7 == 0:
            amax = np.float32(0)
        oracle.update_scale(a, amax, ALGO_MOST_RECENT, E5M2)
        oracle.update_scale(b, amax, ALGO_MAX, E5M2)
        assert a.scale[0] == b.scale[0] and a.scale_inv[0] == b.scale_inv[0]


@pytest.mark.parametrize("fmt,fmax", [(E4M3, 448.0), (E5M2, 57344.0)])
def test_scale_closed_form(fmt, fmax):
    rng = np.random.default_rng(11)
    for _ in range(200):
        amax = np.float32(abs(rng.standard_normal()) * 10.0 ** rng.integers(-6, 6))
        st = oracle.ScaleState(1)
        oracle.update_scale(st, amax, ALGO_MAX, fmt)
        want = np.float32(fmax) / amax
        assert st.scale[0] == want
        assert st.scale_inv[0] == np.float32(1) / want
        # margin m divides by 2^m exactly
        st2 = oracle.ScaleState(1)
        oracle.update_scale(st2, amax, ALGO_MAX, fmt, margin=3)
        assert st2.scale[0] == want / np.float32(8)


def test_pow2_scale_for_power_of_two_amax():
    # 448 / 2^k = 1.75 * 2^(8-k): the power-of-two scale is 2^(8-k), and
    # 57344 / 2^k = 1.75 * 2^(15-k) gives 2^(15-k)
    for k in range(-20, 21):
        for fmt, top in ((E4M3, 8), (E5M2, 15)):
            st = oracle.ScaleState(1)
            oracle.update_scale(st, np.float32(2.0 ** k), ALGO_MAX, fmt, pow2=True)
            assert st.scale[0] == np.float32(2.0 ** (top - k))
            assert st.scale_inv[0] == np.float32(2.0 ** (k - top))


def test_zero_and_nonfinite_amax_keep_previous_scale():
    st = oracle.ScaleState(1)
    oracle.update_scale(st, 2.0, ALGO_MAX, E4M3)
    assert st.scale[0] == 224
    for bad in (0.0, np.inf, np.nan):
        oracle.update_scale(st, bad, ALGO_MAX, E4M3)
        assert st.scale[0] == 224 and st.scale_inv[0] == np.float32(1 / 224)
    fresh = oracle.ScaleState(4)
    oracle.update_scale(fresh, 0.0, ALGO_MAX, E4M3)
    assert fresh.scale[0] == 1 and fresh.scale_inv[0] == 1


def test_scale_clamped_to_normal_range():
    # smallest positive bf16 (a subnormal) drives 448/amax past FLT_MAX
    tiny = oracle.bf16_to_f32(np.array([1], np.uint16))[0]
    st = oracle.ScaleState(1)
    oracle.update_scale(st, tiny, ALGO_MAX, E4M3)
    assert st.scale[0] == FLT_MAX
    assert st.scale_inv[0] == np.float32(1) / FLT_MAX
    st = oracle.ScaleState(1)
    oracle.update_scale(st, tiny, ALGO_MAX, E4M3, pow2=True)
    assert st.scale[0] == np.float32(2.0 ** 127)
    # a huge amax with a large margin is floored at the smallest normal
    st = oracle.ScaleState(1)
    oracle.update_scale(st, np.float32(3e38), ALGO_MAX, E4M3, margin=60)
    assert st.scale[0] == FLT_MIN


def _bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_single_block_equals_per_tensor_quantize():
    rng = np.random.default_rng(5)
    for block_rows, shape in ((128, (128, 128)), (1, (1, 128))):
        for fmt in (E4M3, E5M2):
            bits = _bits(rng.standard_normal(shape) * 0.37)
            q, sinv = oracle.block_quantize(bits, fmt, block_rows)
            a = oracle.amax(bits)
            s = np.float32(oracle.fp8_max(fmt)) / a
            qref, _ = oracle.quantize(bits, fmt, s)
            assert np.array_equal(q, qref)
            assert sinv.shape == (1, 1) and sinv[0, 0] == np.float32(1) / s


def test_block_geometry_and_zero_blocks():
    rng = np.random.default_rng(9)
    rows, cols = 256, 384
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    # give each 128x128 tile its own magnitude; zero one tile
    mags = np.array([[1, 10, 100], [0.01, 0, 1000]], np.float32)
    x *= np.kron(mags, np.ones((128, 128), np.float32))
    bits = _bits(x)
    q, sinv = oracle.block_quantize(bits, E4M3, 128)
    assert sinv.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            tile = bits[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            a = oracle.amax(tile)
            s = np.float32(1) if a == 0 else np.float32(448) / a
            assert sinv[bi, bj] == np.float32(1) / s
            qt, _ = oracle.quantize(tile, E4M3, s)
            assert np.array_equal(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], qt)
    assert sinv[1, 1] == 1 and not (q[128:, 128:256] & 0x7F).any()   # +-0 only
    # 1x128: one scale per row segment
    q1, s1 = oracle.block_quantize(bits, E5M2, 1)
    assert s1.shape == (rows, 3)
    r, bj = 200, 2
    seg = bits[r:r + 1, bj * 128:(bj + 1) * 128]
    s = np.float32(57344) / oracle.amax(seg)
    assert s1[r, bj] == np.float32(1) / s
    assert np.array_equal(q1[r:r + 1, bj * 128:(bj + 1) * 128], oracle.quantize(seg, E5M2, s)[0])


def test_block_pow2_scales_are_powers_of_two():
    rng = np.random.default_rng(2)
    bits = _bits(rng.standard_normal((128, 256)) * 5)
    _, sinv = oracle.block_quantize(bits, E4M3, 1, pow2=True)
    m, e = np.frexp(sinv)
    assert (m == 0.5).all()


def test_row_quantize_rows_are_per_tensor_casts():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((7, 300)).astype(np.float32) * (10.0 ** rng.integers(-3, 3, (7, 1)))
    x[4] = 0
    bits = _bits(x)
    for fmt, fmax in ((E4M3, 448.0), (E5M2, 57344.0)):
        q, sinv = oracle.row_quantize(bits, fmt)
        for i in range(7):
            a = oracle.amax(bits[i])
            s = np.float32(1) if a == 0 else np.float32(fmax) / a
            assert sinv[i] == np.float32(1) / s
            assert np.array_equal(q[i], oracle.quantize(bits[i:i + 1], fmt, s)[0][0])
