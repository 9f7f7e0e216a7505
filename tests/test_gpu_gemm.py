"""GPU parity of the tcgen05 FP8 GEMMs (per-tensor and block-scaled) against
the CPU oracle's fp64 GEMM: within |gpu - oracle| <= 2e-3 * sum|a b| s_a s_b
per element, and exactly equal where every partial sum is representable."""
import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
from tests.helpers import assert_gemm_bound

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    F.build()
    F.lib()
    yield
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0


def _codes(rng, shape, fmt, std=1.0):
    """Realistic FP8 operand: N(0, std^2) values cast with a per-tensor scale."""
    v = rng.standard_normal(shape).astype(np.float32) * std
    b = (v.view(np.uint32) >> 16).astype(np.uint16)
    s = np.float32(oracle.fp8_max(fmt)) / oracle.amax(b)
    q, _ = oracle.quantize(b, fmt, s)
    return q, np.float32(1) / s


def _t(a, dtype=torch.uint8):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _s(v):
    return torch.tensor(np.asarray(v, np.float32).reshape(-1), device=DEV)


SHAPES = [(128, 256, 128), (200, 336, 304), (1, 16, 16), (384, 512, 1024), (129, 272, 4000),
          (256, 768, 2048), (640, 1280, 256)]
FORMATS = [(F.E4M3, F.E4M3), (F.E5M2, F.E4M3), (F.E4M3, F.E5M2), (F.E5M2, F.E5M2)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fa,fb", FORMATS)
def test_tensor_scaled_bf16(M, N, K, fa, fb):
    rng = np.random.default_rng(M + 7 * N + 13 * K + fa * 3 + fb)
    A, sa = _codes(rng, (M, K), fa)
    B, sb = _codes(rng, (N, K), fb, 0.02)
    D = F.fp8_gemm(_t(A), fa, _t(B), fb, _s(sa), _s(sb))
    Do, Dabs = oracle.gemm(A, fa, B, fb, sa, sb)
    assert_gemm_bound(D, Do, Dabs, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(200, 336, 304), (256, 512, 2048), (1000, 272, 640)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_tensor_scaled_f32_accumulate(M, N, K, accumulate):
    rng = np.random.default_rng(M * N + K)
    A, sa = _codes(rng, (M, K), F.E5M2)
    B, sb = _codes(rng, (N, K), F.E4M3)
    prev = rng.standard_normal((M, N)).astype(np.float32)
    D = _t(prev, torch.float32)
    F.fp8_gemm(_t(A), F.E5M2, _t(B), F.E4M3, _s(sa), _s(sb), out=F.OUT_F32, D=D,
               accumulate=accumulate)
    Do, Dabs = oracle.gemm(A, F.E5M2, B, F.E4M3, sa, sb)
    if accumulate:
        assert_gemm_bound(D, Do + prev, Dabs, prev=prev)
    else:
        assert_gemm_bound(D, Do, Dabs)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 512, 4096), (64, 48, 1040)])
def test_exact_integer_products(M, N, K):
    """Small-integer codes and power-of-two scales: every partial sum is an
    integer below 2^24, so the FP32 result must equal the oracle exactly."""
    rng = np.random.default_rng(K)
    ai = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    bi = rng.integers(-4, 5, size=(N, K)).astype(np.float32)
    A = oracle.encode(ai, F.E4M3)
    B = oracle.encode(bi, F.E5M2)
    D = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E5M2, _s(0.5), _s(4.0), out=F.OUT_F32)
    want = (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float64) * 2.0
    assert np.array_equal(D.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("M,N,K", [(2048, 256, 256), (1152, 512, 128), (4864, 128, 64),
                                   (128, 4864, 64), (1040, 1040, 96), (4864, 512, 64),
                                   (5120, 512, 64)])
def test_one_wave_tile_order(M, N, K):
    """Problems whose 128 x 64 (else 128 x 128) tiles fit in one wave run on
    the single-CTA kernel with those tiles, many tiles along M or N: every
    tile lands where its operand rows came from.  Small-integer codes make
    the FP32 result exact, so a tile written to another tile's place cannot
    pass.  On a 152-SM GPU the first four shapes take 64-column tiles, the
    next two 128-column tiles (1040 x 1040 just past one wave of 64-column
    ones, 4864 x 512 exactly one wave of 128-column ones) and the last the
    CTA pairs (160 tiles of 128 x 128), so every kernel runs at a boundary."""
    rng = np.random.default_rng(M + N + K)
    ai = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    bi = rng.integers(-4, 5, size=(N, K)).astype(np.float32)
    A = oracle.encode(ai, F.E4M3)
    B = oracle.encode(bi, F.E4M3)
    want = (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float64) * 0.25
    D = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E4M3, _s(0.5), _s(0.5), out=F.OUT_F32)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), want)
    # bf16 output: the exact product rounded once (torch's cast rounds to nearest even)
    Db = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E4M3, _s(0.5), _s(0.5))
    wb = torch.from_numpy(want.astype(np.float32)).bfloat16()
    assert torch.equal(Db.cpu().view(torch.int16), wb.view(torch.int16))


def test_degenerate_shapes():
    A = torch.zeros(0, 64, dtype=torch.uint8, device=DEV)
    B = torch.zeros(32, 64, dtype=torch.uint8, device=DEV)
    D = F.fp8_gemm(A, F.E4M3, B, F.E4M3, _s(1.0), _s(1.0))
    assert D.shape == (0, 32)
    A = torch.zeros(16, 0, dtype=torch.uint8, device=DEV)
    B = torch.zeros(32, 0, dtype=torch.uint8, device=DEV)
    D = torch.full((16, 32), 7.0, dtype=torch.float32, device=DEV)
    F.fp8_gemm(A, F.E4M3, B, F.E4M3, _s(1.0), _s(1.0), out=F.OUT_F32, D=D)
    assert (D == 0).all()
    D.fill_(7.0)
    F.fp8_gemm(A, F.E4M3, B, F.E4M3, _s(1.0), _s(1.0), out=F.OUT_F32, D=D, accumulate=True)
    assert (D == 7).all()


MN_LAYOUTS = [F.LAYOUT_B_KN, F.LAYOUT_A_KM, F.LAYOUT_KM_KN]


def _stored(A, B, layout):
    """A [M x K] and B [N x K] as fp8_gemm reads them under `layout`."""
    return (_t(A.T if layout & F.LAYOUT_A_KM else A), _t(B.T if layout & F.LAYOUT_B_KN else B))


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (304, 272, 400), (48, 80, 1040),
                                   (640, 768, 1152), (1024, 512, 4096)])
@pytest.mark.parametrize("layout", MN_LAYOUTS)
def test_mn_major_layouts(M, N, K, layout):
    """Operands stored [K x M] / [K x N] (read MN-major by the tensor core):
    within the oracle bound, and from 256 rows on bit-identical to the same
    codes in the TN layout (the same CTA-pair kernel, the same K order)."""
    rng = np.random.default_rng(M + 3 * N + 5 * K + layout)
    A, sa = _codes(rng, (M, K), F.E5M2)
    B, sb = _codes(rng, (N, K), F.E4M3, 0.02)
    a, b = _stored(A, B, layout)
    D = F.fp8_gemm(a, F.E5M2, b, F.E4M3, _s(sa), _s(sb), layout=layout)
    Do, Dabs = oracle.gemm(A, F.E5M2, B, F.E4M3, sa, sb)
    assert_gemm_bound(D, Do, Dabs, what=f"layout {layout} {M}x{N}x{K}")
    if M >= 256:
        ref = F.fp8_gemm(_t(A), F.E5M2, _t(B), F.E4M3, _s(sa), _s(sb))
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (304, 400, 1040), (32, 16, 272)])
@pytest.mark.parametrize("layout", MN_LAYOUTS)
def test_mn_major_exact_integer_products(M, N, K, layout):
    """Small-integer codes in every layout: every partial sum is an exact
    integer, so a misplaced element anywhere (a wrong stride, a swizzle or
    K-step error) changes the FP32 result."""
    rng = np.random.default_rng(K + layout)
    ai = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    bi = rng.integers(-4, 5, size=(N, K)).astype(np.float32)
    a, b = _stored(oracle.encode(ai, F.E4M3), oracle.encode(bi, F.E5M2), layout)
    D = F.fp8_gemm(a, F.E4M3, b, F.E5M2, _s(0.5), _s(4.0), out=F.OUT_F32, layout=layout)
    want = (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float64) * 2.0
    assert np.array_equal(D.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("layout", MN_LAYOUTS)
@pytest.mark.parametrize("ga,gb,out,acc", [(F.GRAN_ROW, F.GRAN_ROW, F.OUT_BF16, False),
                                           (F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_F32, True),
                                           (F.GRAN_ROW, F.GRAN_TENSOR, F.OUT_F32, False)])
def test_mn_major_row_scales_and_f32(layout, ga, gb, out, acc):
    """Per-row factors and the FP32 (accumulating) epilogue with MN-major
    operands: the factors index output rows and columns, not storage."""
    M, N, K = 512, 384, 640
    rng = np.random.default_rng(layout + 10 * ga + 100 * out)
    A, _ = _codes(rng, (M, K), F.E4M3)
    B, _ = _codes(rng, (N, K), F.E4M3, 0.02)
    sa = (rng.random(M if ga == F.GRAN_ROW else 1) + 0.5).astype(np.float32)
    sb = (rng.random(N if gb == F.GRAN_ROW else 1) + 0.5).astype(np.float32)
    a, b = _stored(A, B, layout)
    prev = rng.standard_normal((M, N)).astype(np.float32)
    D = _t(prev, torch.float32) if out == F.OUT_F32 else None
    D = F.fp8_gemm(a, F.E4M3, b, F.E4M3, _s(sa), _s(sb), ga=ga, gb=gb, out=out, D=D,
                   accumulate=acc, layout=layout)
    Do, Dabs = oracle.gemm(A, F.E4M3, B, F.E4M3, sa, sb, ga, gb)
    if acc:
        assert_gemm_bound(D, Do + prev, Dabs, prev=prev)
    else:
        assert_gemm_bound(D, Do, Dabs)


def _block_operand(rng, shape, fmt, gran, std=1.0):
    v = rng.standard_normal(shape).astype(np.float32) * std
    v *= np.abs(rng.standard_t(3, size=(shape[0], 1))).astype(np.float32)
    b = (v.view(np.uint32) >> 16).astype(np.uint16)
    if gran == F.GRAN_TENSOR:
        s = np.float32(oracle.fp8_max(fmt)) / oracle.amax(b)
        return oracle.quantize(b, fmt, s)[0], np.array([1 / s], np.float32)
    return oracle.block_quantize(b, fmt, 1 if gran == F.GRAN_1x128 else 128)


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (200, 384, 1024), (128, 128, 128),
                                   (512, 640, 2048)])
@pytest.mark.parametrize("ga,gb", [(F.GRAN_1x128, F.GRAN_128x128),
                                   (F.GRAN_128x128, F.GRAN_128x128),
                                   (F.GRAN_TENSOR, F.GRAN_128x128),
                                   (F.GRAN_1x128, F.GRAN_TENSOR),
                                   (F.GRAN_1x128, F.GRAN_1x128)])
def test_block_scaled(M, N, K, ga, gb):
    if ga == F.GRAN_128x128 and M % 128:
        pytest.skip("128x128 scales on A need M % 128 == 0")
    rng = np.random.default_rng(M + N + K + ga * 10 + gb)
    A, sa = _block_operand(rng, (M, K), F.E4M3, ga)
    B, sb = _block_operand(rng, (N, K), F.E4M3, gb, 0.02)
    for out in (F.OUT_BF16, F.OUT_F32):
        D = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E4M3, _s(sa), _s(sb), ga, gb, out=out)
        Do, Dabs = oracle.gemm(A, F.E4M3, B, F.E4M3, sa, sb, ga, gb)
        assert_gemm_bound(D, Do, Dabs, what=f"block {M}x{N}x{K} out={out}")


def test_block_scaled_exact():
    """Integer codes with power-of-two block factors: exact in FP32."""
    rng = np.random.default_rng(3)
    M, N, K = 256, 384, 1024
    ai = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    bi = rng.integers(-3, 4, size=(N, K)).astype(np.float32)
    sa = (2.0 ** rng.integers(-3, 4, size=(M, K // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(-3, 4, size=(N // 128, K // 128))).astype(np.float32)
    A, B = oracle.encode(ai, F.E4M3), oracle.encode(bi, F.E4M3)
    D = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E4M3, _s(sa), _s(sb), F.GRAN_1x128, F.GRAN_128x128,
                   out=F.OUT_F32)
    Do, _ = oracle.gemm(A, F.E4M3, B, F.E4M3, sa, sb, F.GRAN_1x128, F.GRAN_128x128)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), Do)


def test_block_scaled_exact_column_scales():
    """1x128 scales on both operands (the wgrad case): every output column has
    its own B factor per K block.  Power-of-two factors: exact in FP32."""
    rng = np.random.default_rng(4)
    M, N, K = 256, 256, 640
    ai = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    bi = rng.integers(-3, 4, size=(N, K)).astype(np.float32)
    sa = (2.0 ** rng.integers(-3, 4, size=(M, K // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(-3, 4, size=(N, K // 128))).astype(np.float32)
    A, B = oracle.encode(ai, F.E5M2), oracle.encode(bi, F.E4M3)
    prev = rng.integers(-8, 8, size=(M, N)).astype(np.float32)
    D = _t(prev, torch.float32)
    F.fp8_gemm(_t(A), F.E5M2, _t(B), F.E4M3, _s(sa), _s(sb), F.GRAN_1x128, F.GRAN_1x128,
               out=F.OUT_F32, D=D, accumulate=True)
    Do, _ = oracle.gemm(A, F.E5M2, B, F.E4M3, sa, sb, F.GRAN_1x128, F.GRAN_1x128)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), Do + prev)


# Power-of-two block factors on both operands (pow2 block casts) run on the
# block-scaled MMA (UE8M0 factors inside the tensor core).  Shapes: one tile,
# ragged M (not a multiple of 256, and below 256), N a multiple of 128 but not
# of 256 (a half-empty last tile column), several tiles and K blocks, and
# more tiles than the grid has CTA pairs.
POW2_SHAPES = [(256, 256, 128), (200, 384, 1024), (128, 128, 256), (384, 640, 2048),
               (1, 128, 128), (1536, 1152, 512), (4096, 4352, 256)]


@pytest.mark.parametrize("M,N,K", POW2_SHAPES)
@pytest.mark.parametrize("ga,gb", [(F.GRAN_1x128, F.GRAN_128x128), (F.GRAN_1x128, F.GRAN_1x128),
                                   (F.GRAN_128x128, F.GRAN_128x128)])
def test_block_scaled_pow2(M, N, K, ga, gb):
    if ga == F.GRAN_128x128 and M % 128:
        pytest.skip("128x128 scales on A need M % 128 == 0")
    rng = np.random.default_rng(M + 3 * N + K + ga * 10 + gb)

    def operand(shape, fmt, gran, std):
        v = rng.standard_normal(shape).astype(np.float32) * std
        v *= np.abs(rng.standard_t(3, size=(shape[0], 1))).astype(np.float32)
        b = (v.view(np.uint32) >> 16).astype(np.uint16)
        return oracle.block_quantize(b, fmt, 1 if gran == F.GRAN_1x128 else 128, pow2=True)

    A, sa = operand((M, K), F.E4M3, ga, 1.0)
    B, sb = operand((N, K), F.E5M2 if gb == F.GRAN_1x128 else F.E4M3, gb, 0.02)
    fb = F.E5M2 if gb == F.GRAN_1x128 else F.E4M3
    Do, Dabs = oracle.gemm(A, F.E4M3, B, fb, sa, sb, ga, gb)
    for out in (F.OUT_BF16, F.OUT_F32):
        D = F.fp8_gemm(_t(A), F.E4M3, _t(B), fb, _s(sa), _s(sb), ga | F.SCALE_POW2,
                       gb | F.SCALE_POW2, out=out)
        assert_gemm_bound(D, Do, Dabs, what=f"pow2 block {M}x{N}x{K} out={out}")


def test_block_scaled_pow2_exact():
    """Integer codes and power-of-two factors spanning 2^-2..2^2 per 128-deep
    block: every partial sum is representable, so the block-scaled MMA must
    reproduce the oracle exactly -- including the FP32 accumulation into D,
    the bias, and the per-column (1x128 on B) factors of the wgrad case."""
    rng = np.random.default_rng(11)
    for M, N, K, ga, gb in [(384, 512, 1024, F.GRAN_1x128, F.GRAN_128x128),
                            (256, 384, 640, F.GRAN_1x128, F.GRAN_1x128),
                            (200, 256, 384, F.GRAN_1x128, F.GRAN_1x128)]:
        ai = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
        bi = rng.integers(-3, 4, size=(N, K)).astype(np.float32)
        sa = (2.0 ** rng.integers(-2, 3, size=(M, K // 128))).astype(np.float32)
        rows_b = N if gb == F.GRAN_1x128 else N // 128
        sb = (2.0 ** rng.integers(-2, 3, size=(rows_b, K // 128))).astype(np.float32)
        A, B = oracle.encode(ai, F.E4M3), oracle.encode(bi, F.E5M2)
        Do, _ = oracle.gemm(A, F.E4M3, B, F.E5M2, sa, sb, ga, gb)
        prev = rng.integers(-8, 8, size=(M, N)).astype(np.float32)
        D = _t(prev, torch.float32)
        F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E5M2, _s(sa), _s(sb), ga | F.SCALE_POW2,
                   gb | F.SCALE_POW2, out=F.OUT_F32, D=D, accumulate=True)
        assert np.array_equal(D.cpu().numpy().astype(np.float64), Do + prev), (M, N, K)
        bias = rng.integers(-4, 5, size=N).astype(np.float32)
        Db = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E5M2, _s(sa), _s(sb), ga | F.SCALE_POW2,
                        gb | F.SCALE_POW2, out=F.OUT_F32,
                        bias=torch.tensor(bias, device=DEV).to(torch.bfloat16))
        assert np.array_equal(Db.cpu().numpy().astype(np.float64), Do + bias[None, :]), (M, N, K)


def test_block_scaled_pow2_equals_promotion():
    """The same power-of-two operands through both block paths (one operand
    flagged runs the per-128-K promotion kernel): equal to within the FP32
    rounding of the two accumulation orders, and both within the bound."""
    rng = np.random.default_rng(12)
    M, N, K = 512, 768, 2048
    v = rng.standard_normal((M, K)).astype(np.float32)
    A, sa = oracle.block_quantize((v.view(np.uint32) >> 16).astype(np.uint16), F.E4M3, 1, pow2=True)
    w = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    B, sb = oracle.block_quantize((w.view(np.uint32) >> 16).astype(np.uint16), F.E4M3, 128, pow2=True)
    args = (_t(A), F.E4M3, _t(B), F.E4M3, _s(sa), _s(sb))
    D_mx = F.fp8_gemm(*args, F.GRAN_1x128 | F.SCALE_POW2, F.GRAN_128x128 | F.SCALE_POW2,
                      out=F.OUT_F32)
    D_pr = F.fp8_gemm(*args, F.GRAN_1x128 | F.SCALE_POW2, F.GRAN_128x128, out=F.OUT_F32)
    Do, Dabs = oracle.gemm(A, F.E4M3, B, F.E4M3, sa, sb, F.GRAN_1x128, F.GRAN_128x128)
    assert_gemm_bound(D_mx, Do, Dabs, what="pow2 MMA")
    assert_gemm_bound(D_pr, Do, Dabs, what="promotion")
    diff = (D_mx - D_pr).abs().cpu().numpy().astype(np.float64)
    assert (diff <= 1e-4 * Dabs + 1e-30).all()


@pytest.mark.parametrize("M,N,K", [(200, 336, 304), (512, 768, 1024), (1, 16, 16)])
@pytest.mark.parametrize("ga,gb", [(F.GRAN_ROW, F.GRAN_ROW), (F.GRAN_ROW, F.GRAN_TENSOR),
                                   (F.GRAN_TENSOR, F.GRAN_ROW)])
@pytest.mark.parametrize("out", [F.OUT_BF16, F.OUT_F32])
def test_row_scaled(M, N, K, ga, gb, out):
    rng = np.random.default_rng(M + N + K + ga + 3 * gb + out)

    def operand(rows, gran, std):
        v = rng.standard_normal((rows, K)).astype(np.float32) * std
        v *= np.abs(rng.standard_t(3, size=(rows, 1))).astype(np.float32)
        b = (v.view(np.uint32) >> 16).astype(np.uint16)
        if gran == F.GRAN_ROW:
            return oracle.row_quantize(b, F.E4M3)
        s = np.float32(448) / oracle.amax(b)
        return oracle.quantize(b, F.E4M3, s)[0], np.array([1 / s], np.float32)

    A, sa = operand(M, ga, 1.0)
    B, sb = operand(N, gb, 0.02)
    D = F.fp8_gemm(_t(A), F.E4M3, _t(B), F.E4M3, _s(sa), _s(sb), ga, gb, out=out)
    Do, Dabs = oracle.gemm(A, F.E4M3, B, F.E4M3, sa, sb, ga, gb)
    assert_gemm_bound(D, Do, Dabs, what=f"row {M}x{N}x{K}")


def _rand_codes(shape, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.randint(0, 0x7C, shape, generator=g, dtype=torch.int32)
    v |= torch.randint(0, 2, shape, generator=g, dtype=torch.int32) << 7
    return v.to(torch.uint8).to(DEV)


@pytest.mark.parametrize("case", ["bwd_like", "ragged", "rowscaled", "fallback_block", "small_m",
                                  "pow2_block_bwd", "bwd_mn_major", "small_m_mn_major",
                                  "bwd_mn_major_large"])
def test_gemm_group_equals_two_gemms(case):
    """fp8_gemm_group gives, bit for bit, the results of two fp8_gemm calls:
    a grouped launch -- the single-CTA kernel when both problems' 128 x 128
    tiles fit in one wave, else CTA pairs (bwd_mn_major_large) -- computes
    every tile exactly as a single launch does; problems it does not take
    fall back to two launches."""
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    if case == "bwd_like":        # dgrad (bf16) and wgrad (FP32, accumulated) of a linear
        M, N, K = 1024, 768, 640
        g1 = dict(A=_rand_codes((M, N), 1), fa=F.E5M2, B=_rand_codes((K, N), 2), fb=F.E4M3,
                  scale_inv_a=one * 2 ** -7, scale_inv_b=one * 2 ** -5)
        g2 = dict(A=_rand_codes((N, M), 3), fa=F.E5M2, B=_rand_codes((K, M), 4), fb=F.E4M3,
                  scale_inv_a=one * 2 ** -7, scale_inv_b=one * 2 ** -6, out=F.OUT_F32,
                  accumulate=True)
    elif case == "ragged":
        g1 = dict(A=_rand_codes((400, 272), 5), fa=F.E4M3, B=_rand_codes((528, 272), 6),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one)
        g2 = dict(A=_rand_codes((300, 1056), 7), fa=F.E4M3, B=_rand_codes((144, 1056), 8),
                  fb=F.E5M2, scale_inv_a=one, scale_inv_b=one * 0.5)
    elif case == "rowscaled":
        s = lambda n, sd: (torch.rand(n, generator=torch.Generator().manual_seed(sd)) + 0.5).to(DEV)
        g1 = dict(A=_rand_codes((512, 256), 9), fa=F.E4M3, B=_rand_codes((384, 256), 10),
                  fb=F.E4M3, scale_inv_a=s(512, 1), scale_inv_b=s(384, 2), ga=F.GRAN_ROW,
                  gb=F.GRAN_ROW)
        g2 = dict(A=_rand_codes((384, 512), 11), fa=F.E5M2, B=_rand_codes((256, 512), 12),
                  fb=F.E4M3, scale_inv_a=s(384, 3), scale_inv_b=s(256, 4), ga=F.GRAN_ROW,
                  gb=F.GRAN_ROW)
    elif case == "fallback_block":
        sa = torch.rand(256, 2, generator=torch.Generator().manual_seed(5)).to(DEV) + 0.5
        sb = torch.rand(2, 2, generator=torch.Generator().manual_seed(6)).to(DEV) + 0.5
        g1 = dict(A=_rand_codes((256, 256), 13), fa=F.E4M3, B=_rand_codes((256, 256), 14),
                  fb=F.E4M3, scale_inv_a=sa, scale_inv_b=sb, ga=F.GRAN_1x128, gb=F.GRAN_128x128)
        g2 = dict(A=_rand_codes((512, 256), 15), fa=F.E4M3, B=_rand_codes((256, 256), 16),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one)
    elif case == "pow2_block_bwd":   # the block backward with power-of-two factors
        M, N, K = 512, 384, 640      # dgrad (bf16) and wgrad (FP32, accumulated)
        p2 = lambda shape, sd: (2.0 ** torch.randint(
            -3, 4, shape, generator=torch.Generator().manual_seed(sd))).float().to(DEV)
        g1 = dict(A=_rand_codes((M, N), 21), fa=F.E5M2, B=_rand_codes((K, N), 22), fb=F.E4M3,
                  scale_inv_a=p2((M, N // 128), 1), scale_inv_b=p2((K // 128, N // 128), 2),
                  ga=F.GRAN_1x128 | F.SCALE_POW2, gb=F.GRAN_128x128 | F.SCALE_POW2)
        g2 = dict(A=_rand_codes((N, M), 23), fa=F.E5M2, B=_rand_codes((K, M), 24), fb=F.E4M3,
                  scale_inv_a=p2((N, M // 128), 3), scale_inv_b=p2((K, M // 128), 4),
                  ga=F.GRAN_1x128 | F.SCALE_POW2, gb=F.GRAN_1x128 | F.SCALE_POW2,
                  out=F.OUT_F32, accumulate=True)
    elif case == "bwd_mn_major":   # dgrad and wgrad reading the forward's codes as stored
        M, N, K = 1024, 768, 640
        dy, w, x = _rand_codes((M, N), 25), _rand_codes((N, K), 26), _rand_codes((M, K), 27)
        g1 = dict(A=dy, fa=F.E5M2, B=w, fb=F.E4M3, scale_inv_a=one * 2 ** -7,
                  scale_inv_b=one * 2 ** -5, layout=F.LAYOUT_B_KN)
        g2 = dict(A=dy, fa=F.E5M2, B=x, fb=F.E4M3, scale_inv_a=one * 2 ** -7,
                  scale_inv_b=one * 2 ** -6, out=F.OUT_F32, accumulate=True,
                  layout=F.LAYOUT_KM_KN)
    elif case == "bwd_mn_major_large":   # 192 + 144 tiles of 128 x 128: the grouped CTA pairs
        M, N, K = 2048, 1536, 1536
        dy, w, x = _rand_codes((M, N), 32), _rand_codes((N, K), 33), _rand_codes((M, K), 34)
        g1 = dict(A=dy, fa=F.E5M2, B=w, fb=F.E4M3, scale_inv_a=one * 2 ** -7,
                  scale_inv_b=one * 2 ** -5, layout=F.LAYOUT_B_KN)
        g2 = dict(A=dy, fa=F.E5M2, B=x, fb=F.E4M3, scale_inv_a=one * 2 ** -7,
                  scale_inv_b=one * 2 ** -6, out=F.OUT_F32, accumulate=True,
                  layout=F.LAYOUT_KM_KN)
    elif case == "small_m_mn_major":   # fewer than 256 rows, MN-major: one grouped launch
        g1 = dict(A=_rand_codes((640, 96), 28), fa=F.E5M2, B=_rand_codes((640, 512), 29),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one, out=F.OUT_F32,
                  layout=F.LAYOUT_KM_KN)
        g2 = dict(A=_rand_codes((128, 640), 30), fa=F.E5M2, B=_rand_codes((640, 256), 31),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one, layout=F.LAYOUT_B_KN)
    else:                          # M < 256: the 1-CTA kernel, two launches
        g1 = dict(A=_rand_codes((128, 256), 17), fa=F.E4M3, B=_rand_codes((256, 256), 18),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one)
        g2 = dict(A=_rand_codes((512, 256), 19), fa=F.E4M3, B=_rand_codes((256, 256), 20),
                  fb=F.E4M3, scale_inv_a=one, scale_inv_b=one)
    prev = None
    if g2.get("out") == F.OUT_F32:
        M2, _, N2 = F._gemm_dims(g2["A"], g2["B"], g2.get("layout", F.LAYOUT_TN))
        prev = torch.randn(M2, N2, device=DEV)
        g2["D"] = prev.clone()
    D1, D2 = F.fp8_gemm_group(g1, g2)
    r1 = F.fp8_gemm(**g1)
    g2b = dict(g2)
    if prev is not None:
        g2b["D"] = prev.clone()
    r2 = F.fp8_gemm(**g2b)
    torch.cuda.synchronize()
    for a, b in ((D1, r1), (D2, r2)):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
