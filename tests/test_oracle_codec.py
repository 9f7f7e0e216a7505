"""Pins of the oracle's FP8 codec and per-tensor quantiser against what the
pages print and what the mathematics and an independent library fix.

Sources: "Mixed Precision LLM Training: The Complete Guide", sections "The
precision formats", "FP8 E4M3", "FP8 E5M2" (bit layouts and ranges) and
"Transformer Engine internals" > "Per-tensor scaling" (scale, then cast).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"e4m3": E4M3, "e5m2": E5M2}
TORCH_FMT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _nan_code(c, fmt):
    if fmt == E4M3:
        return (c & 0x7F) == 0x7F
    return (c & 0x7C) == 0x7C and (c & 0x3) != 0


def _inf_code(c, fmt):
    return fmt == E5M2 and (c & 0x7F) == 0x7C


def test_format_constants_from_pages():
    # golden: the ranges printed in the pages' format table
    for line in open(os.path.join(GOLDEN, "fp8_format_constants.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, e_bits, m_bits, vmax, log2_min = line.split()
        fmt = FMT[name]
        assert oracle.fp8_max(fmt) == float(vmax)
        codes = np.arange(256, dtype=np.uint8)
        vals = oracle.decode(codes, fmt)
        finite = vals[np.isfinite(vals)]
        assert finite.max() == float(vmax)
        assert finite[finite > 0].min() == 2.0 ** int(log2_min)
        # 1 sign + e exponent + m mantissa bits = 8
        assert 1 + int(e_bits) + int(m_bits) == 8


def test_decode_matches_torch_float8_for_every_code():
    # an independent library decode of all 256 codes of each format
    codes = np.arange(256, dtype=np.uint8)
    for fmt, tdt in TORCH_FMT.items():
        ours = oracle.decode(codes, fmt)
        ref = torch.from_numpy(codes).view(tdt).to(torch.float64).numpy()
        for c in range(256):
            if _nan_code(c, fmt):
                assert math.isnan(ours[c]) and math.isnan(ref[c]), c
            else:
                assert ours[c] == ref[c] and np.signbit(ours[c]) == np.signbit(ref[c]), c


def test_nan_and_inf_code_sets():
    codes = np.arange(256, dtype=np.uint8)
    v4 = oracle.decode(codes, E4M3)
    assert [c for c in range(256) if math.isnan(v4[c])] == [0x7F, 0xFF]
    assert not np.isinf(v4).any()            # e4m3 "fn": no infinities
    v5 = oracle.decode(codes, E5M2)
    assert sorted(c for c in range(256) if np.isinf(v5[c])) == [0x7C, 0xFC]
    assert sum(math.isnan(v) for v in v5) == 6


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_every_code_round_trips(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(codes, fmt)
    keep = np.isfinite(vals)
    back = oracle.encode(vals[keep].astype(np.float32), fmt)
    assert np.array_equal(back, codes[keep])


def test_rne_ties_and_saturation_golden():
    for line in open(os.path.join(GOLDEN, "rne_ties.txt")):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        fmt = FMT[parts[0]]
        x = np.float32(float(parts[1]))
        want = float(parts[2])
        got = oracle.decode(oracle.encode(np.array([x]), fmt), fmt)[0]
        assert got == want and np.signbit(got) == np.signbit(want), line


def test_nan_encodes_to_canonical_nan():
    for fmt in (E4M3, E5M2):
        c = oracle.encode(np.array([np.nan, -np.nan], np.float32), fmt)
        assert list(c) == [0x7F, 0x7F]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("scale", [1.0, 0.5, 3.0, 448.0 / 3.0, 1e-3, 2.0 ** 20])
def test_quantize_matches_torch_cast_in_range(fmt, scale):
    # every bf16 bit pattern, multiplied by the scale in fp32 and cast; torch's
    # float8 cast is round-to-nearest-even and agrees wherever no saturation
    # is involved (it does not saturate out-of-range values)
    bits = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    q, qt = oracle.quantize(bits, fmt, scale, transpose=True)
    assert np.array_equal(qt, q.T)
    with np.errstate(invalid="ignore", over="ignore"):
        v = oracle.bf16_to_f32(bits) * np.float32(scale)
    ref = torch.from_numpy(v).to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
    inrange = np.isfinite(v) & (np.abs(v) <= oracle.fp8_max(fmt))
    assert np.array_equal(q[inrange], ref[inrange])
    # beyond the range: saturate to +-max with the sign kept
    over = np.isfinite(v) & (np.abs(v) > oracle.fp8_max(fmt))
    mx = 0x7E if fmt == E4M3 else 0x7B
    assert np.array_equal(q[over] & 0x7F, np.full(over.sum(), mx, np.uint8))
    assert np.array_equal(q[over] >> 7, (v[over] < 0).astype(np.uint8))
    assert (q[np.isnan(v)] == 0x7F).all()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_representable_values_survive_quantise_dequantise(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(codes, fmt)
    finite = vals[np.isfinite(vals)].astype(np.float32)
    # every FP8 value is a bf16 value; scale by 2^k and undo with 2^-k
    for k in (0, 3, -4):
        bits = (finite.astype(np.float32) * np.float32(2.0 ** -k)).view(np.uint32) >> 16
        bits = bits.astype(np.uint16).reshape(1, -1)
        q, _ = oracle.quantize(bits, fmt, 2.0 ** k)
        back = oracle.decode(q, fmt).reshape(-1)
        assert np.array_equal(back, finite.astype(np.float64))


def test_bf16_amax_matches_numpy():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(10007).astype(np.float32) * 3
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    ref = np.abs(oracle.bf16_to_f32(bits)).max()
    assert oracle.amax(bits) == ref
    assert oracle.amax(np.zeros(5, np.uint16)) == 0.0
    assert oracle.amax(np.array([0x8000, 0x0000], np.uint16)) == 0.0   # -0, +0
    assert oracle.amax(np.array([0xFF80, 0x3F80], np.uint16)) == np.inf   # -inf
    assert math.isnan(oracle.amax(np.array([0x3F80, 0x7FC1, 0xFF80], np.uint16)))


def test_cast_counts_golden_cases():
    # hand-picked values around the E4M3 edges with scale 1:
    #   448 (max, not saturated), 464 and 1e30 and -inf (saturated), nan (neither),
    #   2^-10 (tie -> 0: flushed), 3*2^-11 (above the tie: 2^-9, kept), 0 and -0 (not counted)
    vals = np.array([448.0, 464.0, 1e30, -np.inf, np.nan, 2.0 ** -10, 3 * 2.0 ** -11, 0.0, -0.0,
                     -2.0 ** -12], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert oracle.cast_counts(bits, E4M3, 1.0) == (2, 3)
    # E5M2: 57344 max; 2^-17 is the tie to zero
    vals = np.array([57344.0, 61440.0, 2.0 ** -17, 2.0 ** -16, 1.0], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert oracle.cast_counts(bits, E5M2, 1.0) == (1, 1)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_cast_counts_match_direct_definition(fmt):
    # every bf16 pattern, several scales: count straight from numpy and torch
    bits = np.arange(65536, dtype=np.uint16)
    for scale in (1.0, 3.0, 1e-3, 2.0 ** 20):
        with np.errstate(invalid="ignore", over="ignore"):
            v = oracle.bf16_to_f32(bits) * np.float32(scale)
        sat = int(np.sum(np.abs(v) > oracle.fp8_max(fmt)))
        # flushed: finite nonzero input whose product rounds to a zero code (torch's RNE cast)
        t = torch.from_numpy(np.where(np.isfinite(v) & (np.abs(v) <= oracle.fp8_max(fmt)), v, 0)
                             .astype(np.float32)).to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
        nz = (bits & 0x7FFF) != 0
        under = int(np.sum(nz & np.isfinite(v) & (np.abs(v) <= oracle.fp8_max(fmt)) & ((t & 0x7F) == 0)))
        assert oracle.cast_counts(bits, fmt, scale) == (under, sat)
