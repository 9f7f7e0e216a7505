"""Seeded randomized parity sweep over the composed paths: random shapes (ragged
where the call allows it), formats, scale granularities, GEMM operand layouts,
recipes, bias and stochastic rounding, each checked against the oracle with the same bars as
the targeted tests -- codes and scales bit-exact, GEMM results within
2e-3 * sum|a b| * s_a * s_b (+ bf16 rounding)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import assert_gemm_bound, bits, f32bits, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    F.build()
    F.lib()
    yield
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0


def _pick(rng, choices):
    return choices[int(rng.integers(len(choices)))]


@pytest.mark.parametrize("case", range(24))
def test_random_casts(case):
    rng = np.random.default_rng(1000 + case)
    gran = _pick(rng, [F.GRAN_TENSOR, F.GRAN_1x128, F.GRAN_128x128, F.GRAN_ROW])
    fmt = _pick(rng, [F.E4M3, F.E5M2])
    transpose = bool(rng.integers(2))
    pow2 = bool(rng.integers(2))
    if gran == F.GRAN_TENSOR:
        rows, cols = 16 * int(rng.integers(1, 40)), 16 * int(rng.integers(1, 40))
    elif gran == F.GRAN_1x128:
        rows = 128 * int(rng.integers(1, 5)) if transpose else int(rng.integers(1, 300))
        cols = 128 * int(rng.integers(1, 5))
    elif gran == F.GRAN_128x128:
        rows, cols = 128 * int(rng.integers(1, 5)), 128 * int(rng.integers(1, 5))
    else:
        rows, cols = 16 * int(rng.integers(1, 40)), 16 * int(rng.integers(1, 40))
    x = synthetic.student_t_rows((rows, cols), 1.0, 3, seed=case) * float(10.0 ** rng.integers(-3, 3))
    x = x.to(torch.bfloat16)
    if gran == F.GRAN_TENSOR:
        sc = np.float32(10.0 ** rng.uniform(-2, 3))
        q, qt, _, am = F.fp8_quantize(x.to(DEV), fmt, scale=torch.tensor([sc], device=DEV),
                                      transpose=transpose, want_amax=True)
        qo, qto = oracle.quantize(bits(x), fmt, sc, transpose=True)
        assert np.array_equal(u8(q), qo)
        if transpose:
            assert np.array_equal(u8(qt), qto)
        assert f32bits(am.cpu().numpy())[0] == f32bits(oracle.amax(bits(x)))
        return
    q, s, qt, st = F.fp8_quantize_blocks(x.to(DEV), fmt, gran, pow2=pow2, transpose=transpose)
    if gran == F.GRAN_ROW:
        qo, so = oracle.row_quantize(bits(x), fmt, pow2)
    else:
        qo, so = oracle.block_quantize(bits(x), fmt, 1 if gran == F.GRAN_1x128 else 128, pow2)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(f32bits(s.cpu().numpy()), f32bits(so))
    if transpose:
        xt = np.ascontiguousarray(bits(x).T)
        if gran == F.GRAN_ROW:
            qto, sto = oracle.row_quantize(xt, fmt, pow2)
        elif gran == F.GRAN_1x128:
            qto, sto = oracle.block_quantize(xt, fmt, 1, pow2)
        else:
            qto, sto = np.ascontiguousarray(qo.T), np.ascontiguousarray(so.T)
        assert np.array_equal(u8(qt), qto)
        assert np.array_equal(f32bits(st.cpu().numpy()), f32bits(sto))


@pytest.mark.parametrize("case", range(16))
def test_random_gemms(case):
    """Random shapes (ragged against the 256 x 256 tiles), operand layouts,
    per-tensor / per-row factors and outputs of fp8_gemm."""
    rng = np.random.default_rng(3000 + case)
    layout = _pick(rng, [F.LAYOUT_TN, F.LAYOUT_B_KN, F.LAYOUT_A_KM, F.LAYOUT_KM_KN])
    M, N, K = (16 * int(rng.integers(1, 48)) for _ in range(3))
    fa, fb = _pick(rng, [F.E4M3, F.E5M2]), _pick(rng, [F.E4M3, F.E5M2])
    ga, gb = _pick(rng, [F.GRAN_TENSOR, F.GRAN_ROW]), _pick(rng, [F.GRAN_TENSOR, F.GRAN_ROW])
    out = _pick(rng, [F.OUT_BF16, F.OUT_F32])
    acc = out == F.OUT_F32 and bool(rng.integers(2))
    g = torch.Generator().manual_seed(case)
    A = torch.randint(0, 0x7C, (M, K), generator=g, dtype=torch.int32)
    B = torch.randint(0, 0x7C, (N, K), generator=g, dtype=torch.int32)
    A = (A | (torch.randint(0, 2, (M, K), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).numpy()
    B = (B | (torch.randint(0, 2, (N, K), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).numpy()
    sa = (rng.random(M if ga == F.GRAN_ROW else 1) * 2 ** -4 + 2 ** -6).astype(np.float32)
    sb = (rng.random(N if gb == F.GRAN_ROW else 1) * 2 ** -4 + 2 ** -6).astype(np.float32)
    a = A.T if layout & F.LAYOUT_A_KM else A
    b = B.T if layout & F.LAYOUT_B_KN else B
    prev = rng.standard_normal((M, N)).astype(np.float32)
    D = torch.from_numpy(prev).to(DEV) if out == F.OUT_F32 else None
    D = F.fp8_gemm(torch.from_numpy(np.ascontiguousarray(a)).to(DEV), fa,
                   torch.from_numpy(np.ascontiguousarray(b)).to(DEV), fb,
                   torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV), ga=ga, gb=gb,
                   out=out, D=D, accumulate=acc, layout=layout)
    Do, Dabs = oracle.gemm(A, fa, B, fb, sa, sb, ga, gb)
    if acc:
        assert_gemm_bound(D, Do + prev, Dabs, prev=prev, what=f"case {case}")
    else:
        assert_gemm_bound(D, Do, Dabs, what=f"case {case}")


@pytest.mark.parametrize("case", range(12))
def test_random_block_gemms(case):
    """Random shapes (M ragged against the 256-row tiles, N against the
    256-column tiles of the fp32-factor kernel), block-scale granularities of
    both operands (1x128, 128x128, per tensor), fp32 or power-of-two factors,
    and bf16 or accumulated FP32 outputs of fp8_gemm."""
    rng = np.random.default_rng(4000 + case)
    N, K = (128 * int(rng.integers(1, 8)) for _ in range(2))
    ga = _pick(rng, [F.GRAN_1x128, F.GRAN_128x128, F.GRAN_TENSOR])
    gb = _pick(rng, [F.GRAN_1x128, F.GRAN_128x128, F.GRAN_TENSOR])
    if ga == gb == F.GRAN_TENSOR:
        gb = F.GRAN_128x128
    M = 128 * int(rng.integers(1, 6)) if ga == F.GRAN_128x128 else 16 * int(rng.integers(1, 40))
    pow2 = ga != F.GRAN_TENSOR and gb != F.GRAN_TENSOR and bool(rng.integers(2))
    fa, fb = _pick(rng, [F.E4M3, F.E5M2]), _pick(rng, [F.E4M3, F.E5M2])
    out = _pick(rng, [F.OUT_BF16, F.OUT_F32])
    acc = out == F.OUT_F32 and bool(rng.integers(2))
    g = torch.Generator().manual_seed(100 + case)
    A = torch.randint(0, 0x7C, (M, K), generator=g, dtype=torch.int32)
    B = torch.randint(0, 0x7C, (N, K), generator=g, dtype=torch.int32)
    A = (A | (torch.randint(0, 2, (M, K), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).numpy()
    B = (B | (torch.randint(0, 2, (N, K), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).numpy()

    def factors(gran, rows):
        shape = {F.GRAN_TENSOR: (1,), F.GRAN_1x128: (rows, K // 128),
                 F.GRAN_128x128: ((rows + 127) // 128, K // 128)}[gran]
        if pow2:
            return (2.0 ** rng.integers(-8, -3, size=shape)).astype(np.float32)
        return (rng.random(shape) * 2 ** -4 + 2 ** -6).astype(np.float32)

    sa, sb = factors(ga, M), factors(gb, N)
    flag = F.SCALE_POW2 if pow2 else 0
    prev = rng.standard_normal((M, N)).astype(np.float32)
    D = torch.from_numpy(prev).to(DEV) if out == F.OUT_F32 else None
    D = F.fp8_gemm(torch.from_numpy(A).to(DEV), fa, torch.from_numpy(B).to(DEV), fb,
                   torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV), ga=ga | flag,
                   gb=gb | flag, out=out, D=D, accumulate=acc)
    Do, Dabs = oracle.gemm(A, fa, B, fb, sa, sb, ga, gb)
    what = f"case {case}: {M}x{N}x{K} ga={ga} gb={gb} pow2={pow2} out={out} acc={acc}"
    if acc:
        assert_gemm_bound(D, Do + prev, Dabs, prev=prev, what=what)
    else:
        assert_gemm_bound(D, Do, Dabs, what=what)


def _orecipe(r):
    return oracle.Recipe(scaling=r.scaling, margin=r.margin, history_len=r.history_len,
                         algo=r.amax_algo, pow2=bool(r.pow2), sr_grad=bool(r.sr_grad))


@pytest.mark.parametrize("case", range(16))
def test_random_linear_steps(case):
    rng = np.random.default_rng(2000 + case)
    scaling = _pick(rng, [F.SCALING_DELAYED, F.SCALING_DYNAMIC, F.SCALING_BLOCK, F.SCALING_ROW])
    mult = 128 if scaling == F.SCALING_BLOCK else 16
    M = 128 * int(rng.integers(1, 5)) if scaling == F.SCALING_BLOCK else 16 * int(rng.integers(1, 40))
    N, K = mult * int(rng.integers(1, 6 if mult == 128 else 40)), mult * int(rng.integers(1, 6 if mult == 128 else 40))
    sr = scaling in (F.SCALING_DELAYED, F.SCALING_DYNAMIC) and bool(rng.integers(2))
    rec = F.Recipe(scaling, margin=int(rng.integers(0, 2)), history_len=int(rng.integers(1, 20)),
                   amax_algo=_pick(rng, [F.AMAX_MAX, F.AMAX_MOST_RECENT]), pow2=bool(rng.integers(2)),
                   sr_grad=sr)
    with_bias = bool(rng.integers(2))
    seed = int(rng.integers(1 << 62))
    transposes = bool(rng.integers(2))   # per-tensor recipes: K-major copies or MN-major reads
    layer = F.Fp8Linear(M, N, K, rec, device=DEV, sr_seed=seed, transposes=transposes)
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec, sr_seed=seed)
    W = synthetic.normal((N, K), 0.02, seed=case)
    b = synthetic.normal((N,), 0.1, seed=case + 1) if with_bias else None
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    db = torch.zeros(N, dtype=torch.float32, device=DEV) if with_bias else None
    dW_o = np.zeros((N, K))
    db_o = np.zeros(N)
    for step in range(3):
        X = synthetic.with_outlier_channels((M, K), 1.0, min(4, K), 50.0, seed=100 * case + step)
        dY = synthetic.student_t((M, N), 3, 1e-3, seed=200 * case + step)
        acc = step > 0
        Y = layer.forward(X.to(DEV), W.to(DEV), bias=None if b is None else b.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW, accumulate_dW=acc, dbias=db)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost, bias=None if b is None else bits(b))
        prev = dW_o.copy()
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost,
                                                       dW_prev=prev if acc else None)
        assert_gemm_bound(Y, Yo, Yabs + 2.0 ** -13 * np.abs(Yo), what=f"Y step {step}")
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, prev=prev if acc else None, what=f"dW step {step}")
        dW_o = dW.cpu().numpy().astype(np.float64)
        if with_bias:
            # fixed-order FP32 column sums: at most 16 + ceil(M/128) chained additions
            s_, sabs = oracle.dbias(bits(dY))
            want = s_ + (db_o if acc else 0.0)
            tol = (18 + (M + 127) // 128) * 2.0 ** -24 * (sabs + np.abs(db_o))
            got = db.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - want) <= tol), f"dbias step {step}"
            db_o = got
    torch.cuda.synchronize()
