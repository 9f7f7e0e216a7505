"""Pins of the oracle's stochastic-rounding cast.

"Mixed Precision LLM Training: The Complete Guide", "Stochastic rounding":
instead of rounding to nearest, round up or down at random with the
probability set by the remainder, which makes the rounding unbiased.  The
random words come from Philox-4x32-10 (Salmon et al., SC'11).

Pins, none of which re-types the oracle's arithmetic:
  * the generator against its published known-answer vectors;
  * each decision against a brute-force search of the FP8 value table (the
    two neighbours of |v| and the exact switching point of the 32-bit draw,
    computed in fp64 from decoded codes);
  * unbiasedness (the property the pages name) over many draws;
  * special values, determinism, and the counter layout's independence of
    the tensor's shape.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import E4M3, E5M2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        got = oracle.philox4x32_10(w[0:4], w[4:6])
        assert [int(v) for v in got] == w[6:10]
        n += 1
    assert n == 3


def _table(fmt):
    """Finite non-negative FP8 values and their codes, ascending."""
    top = 0x7E if fmt == E4M3 else 0x7B
    codes = np.arange(top + 1, dtype=np.uint8)
    return oracle.decode(codes, fmt), codes


def _expected(v, fmt, r):
    """Brute force: the two table neighbours of |v| and the draw threshold."""
    vals, codes = _table(fmt)
    a = abs(float(np.float32(v)))
    sign = 0x80 if np.signbit(np.float32(v)) else 0
    if a >= vals[-1]:
        return sign | int(codes[-1])
    k = int(np.searchsorted(vals, a, side="right")) - 1      # vals[k] <= a < vals[k+1]
    lo, hi = vals[k], vals[k + 1]
    if a == lo:
        return sign | int(codes[k])
    f = (a - lo) / (hi - lo)                                 # exact: dyadic values
    t = int(np.floor(f * 2.0 ** 32))
    return sign | int(codes[k + 1] if r < t else codes[k])


def _sample_values(seed, n=1500):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, n)
    ex = rng.integers(-30, 20, n)
    v = (mant * 2.0 ** ex * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    extra = np.array([2.0 ** -6, 2.0 ** -9, 2.0 ** -14, 2.0 ** -16, 3 * 2.0 ** -10, 2.0 ** -17,
                      448.0, 449.0, 479.0, 480.0, 500.0, 57344.0, 60000.0, 61440.0, 1e9,
                      1e-40, 1.4e-45, 0.3, 0.1, 1.0, 1.0625, 1.125 + 2.0 ** -20],
                     dtype=np.float32)
    return np.concatenate([v, extra, -extra])


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decisions_match_brute_force(fmt):
    vals, _ = _table(fmt)
    rng = np.random.default_rng(11 + fmt)
    for v in _sample_values(fmt):
        a = abs(float(v))
        # the switching point of the draw, where one exists
        probes = [0, 1, 0x7FFFFFFF, 0xFFFFFFFF, int(rng.integers(0, 2 ** 32))]
        if 0 < a < vals[-1]:
            k = int(np.searchsorted(vals, a, side="right")) - 1
            if a != vals[k]:
                t = int(np.floor((a - vals[k]) / (vals[k + 1] - vals[k]) * 2.0 ** 32))
                probes += [max(t - 1, 0), t, min(t + 1, 2 ** 32 - 1)]
        for r in probes:
            assert oracle.encode_sr(v, fmt, r) == _expected(v, fmt, r), (float(v), r)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_grid_values_never_move(fmt):
    vals, codes = _table(fmt)
    for val, c in zip(vals, codes):
        for r in (0, 1, 0xFFFFFFFF, 0x12345678):
            assert oracle.encode_sr(val, fmt, r) == c
            if val != 0:
                assert oracle.encode_sr(-val, fmt, r) == (0x80 | int(c))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_special_values(fmt):
    top = 0x7E if fmt == E4M3 else 0x7B
    for r in (0, 0xFFFFFFFF):
        assert oracle.encode_sr(np.nan, fmt, r) == 0x7F
        assert oracle.encode_sr(np.inf, fmt, r) == top
        assert oracle.encode_sr(-np.inf, fmt, r) == 0x80 | top
        assert oracle.encode_sr(0.0, fmt, r) == 0x00
        assert oracle.encode_sr(-0.0, fmt, r) == 0x80
    # r = 2^32 - 1 truncates toward zero, r = 0 rounds away from zero
    assert oracle.encode_sr(0.3, E4M3, 0xFFFFFFFF) == oracle.encode(np.array([0.28125], np.float32), E4M3)[0]
    assert oracle.encode_sr(0.3, E4M3, 0) == oracle.encode(np.array([0.3125], np.float32), E4M3)[0]


def _bf16_const(value, shape):
    import torch
    x = torch.full(shape, value, dtype=torch.float32).to(torch.bfloat16)
    v = float(x[0, 0].float())
    return x.contiguous().view(torch.int16).numpy().view(np.uint16), v


@pytest.mark.parametrize("fmt,value,scale", [(E4M3, 0.3, 1.0), (E4M3, 0.0041, 1.0),
                                             (E4M3, 1.7, 100.0), (E5M2, 0.3, 1.0),
                                             (E5M2, 3.0e-6, 1.0)])
def test_unbiased(fmt, value, scale):
    """E[decode(q)] = fp32(x) * scale within the sampling error, while round to
    nearest keeps a fixed bias."""
    xb, v = _bf16_const(value, (256, 1024))
    target = float(np.float32(v) * np.float32(scale))
    q, _ = oracle.quantize_sr(xb, fmt, scale, seed=1234, offset=7)
    d = oracle.decode(q.ravel(), fmt)
    vals, _ = _table(fmt)
    k = int(np.searchsorted(vals, target, side="right")) - 1
    lo, hi = vals[k], vals[k + 1]
    assert set(np.unique(d)) <= {lo, hi}
    f = (target - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(f * (1 - f) / d.size)
    assert abs(d.mean() - target) < 5 * sigma + 1e-300
    rne = oracle.decode(oracle.quantize(xb[:1, :1], fmt, scale)[0].ravel(), fmt)[0]
    assert abs(rne - target) > 20 * sigma


def test_counter_layout_is_shape_independent_and_transposes():
    rng = np.random.default_rng(3)
    xb = (rng.standard_normal((48, 80)) * 3).astype(np.float32)
    import torch
    xb = torch.from_numpy(xb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, qt = oracle.quantize_sr(xb, E4M3, 2.0, seed=99, offset=5, transpose=True)
    assert np.array_equal(qt, q.T)
    # same elements, other shape: codes follow the row-major element index
    q2, _ = oracle.quantize_sr(xb.reshape(80, 48), E4M3, 2.0, seed=99, offset=5)
    assert np.array_equal(q2.reshape(48, 80), q)
    q3, _ = oracle.quantize_sr(xb.reshape(1, -1), E4M3, 2.0, seed=99, offset=5)
    assert np.array_equal(q3.reshape(48, 80), q)
    # element i uses word i % 4 of the block of counter i // 4
    for i in (0, 1, 2, 3, 4, 1001, 3839):
        r = oracle.philox4x32_10([i // 4, 0, 5, 0], [99, 0])[i % 4]
        v = np.float32(oracle.bf16_to_f32(xb.ravel()[i:i + 1])[0] * np.float32(2.0))
        assert q.ravel()[i] == oracle.encode_sr(v, E4M3, int(r))


def test_seed_and_offset_select_independent_draws():
    xb, _ = _bf16_const(0.3, (64, 256))
    a, _ = oracle.quantize_sr(xb, E4M3, 1.0, seed=1, offset=0)
    b, _ = oracle.quantize_sr(xb, E4M3, 1.0, seed=1, offset=0)
    c, _ = oracle.quantize_sr(xb, E4M3, 1.0, seed=2, offset=0)
    d, _ = oracle.quantize_sr(xb, E4M3, 1.0, seed=1, offset=1)
    e, _ = oracle.quantize_sr(xb, E4M3, 1.0, seed=1 << 40, offset=1 << 40)
    assert np.array_equal(a, b)
    for o in (c, d, e):
        agree = np.mean(a == o)
        # independent draws with P(up) = 0.6: agreement 0.6^2 + 0.4^2 = 0.52
        assert 0.47 < agree < 0.57


def test_linear_backward_with_stochastic_gradient_cast():
    """recipe.sr_grad: backward call t casts dY with quantize_sr(seed, t); the
    dequantised codes average to the scaled gradient over many calls."""
    import torch
    M, N, K = 32, 64, 32
    X = torch.randn(M, K).to(torch.bfloat16)
    W = (torch.randn(N, K) * 0.02).to(torch.bfloat16)
    dY = torch.full((M, N), 0.3e-3, dtype=torch.float32)
    dY[0, 0] = 1e-3                       # sets the amax: the rest falls between grid points
    dY = dY.to(torch.bfloat16)
    b = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    rec = oracle.Recipe(scaling=oracle.SCALING_DYNAMIC, sr_grad=True)
    st = oracle.LinearState(rec, sr_seed=42)
    codes = []
    for t in range(40):
        oracle.linear_fwd(b(X), b(W), rec, st)
        oracle.linear_bwd(b(dY), rec, st)
        want, _ = oracle.quantize_sr(b(dY), E5M2, st.roles[2].scale[0], 42, t)
        assert np.array_equal(st.dy_q, want)
        codes.append(oracle.decode(st.dy_q.ravel()[1:], E5M2))
    assert st.sr_counter == 40
    v = float(np.float32(float(dY[0, 1].float())) * np.float32(st.roles[2].scale[0]))
    mean = np.mean(codes)
    vals, _ = _table(E5M2)
    k = int(np.searchsorted(vals, v, side="right")) - 1
    lo, hi = vals[k], vals[k + 1]
    f = (v - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(f * (1 - f) / (40 * (M * N - 1)))
    assert 0.05 < f < 0.95 and abs(mean - v) < 5 * sigma
