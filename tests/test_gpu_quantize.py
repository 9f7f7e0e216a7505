"""GPU parity of the memory-bound kernels (amax, scale update, per-tensor
cast with fused transpose and amax, 1x128 / 128x128 block casts) against
the CPU oracle: every byte, amax and scale bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import bits, f32bits, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    F.build()
    F.lib()
    yield
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0


def _all_bf16_patterns():
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(256, 256)


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("scale", [1.0, 0.5, 3.0, 448.0 / 3.0, 1e-3, 2.0 ** 20, 3.4e38, 1.2e-38])
@pytest.mark.parametrize("transpose", [False, True])
def test_every_bf16_pattern(fmt, scale, transpose):
    x = _all_bf16_patterns()
    s = torch.tensor([scale], dtype=torch.float32, device=DEV)
    q, qt, _, am = F.fp8_quantize(x.to(DEV), fmt, scale=s, transpose=transpose, want_amax=True)
    qo, qto = oracle.quantize(bits(x), fmt, np.float32(scale), transpose=True)
    got = u8(q)
    bad = np.argwhere(got != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, e.g. x bits {bits(x)[tuple(bad[0])]:#06x}: gpu {got[tuple(bad[0])]:#04x} oracle {qo[tuple(bad[0])]:#04x}"
    if transpose:
        assert np.array_equal(u8(qt), qto)
    assert f32bits(am.cpu().numpy())[0] == f32bits(oracle.amax(bits(x)))


@pytest.mark.parametrize("rows,cols,transpose", [
    (3, 37, False), (1, 1, False), (1, 15, False), (17, 16, False), (1008, 48, True),
    (16, 16, True), (144, 400, True), (160, 272, True), (0, 64, False), (0, 0, True),
    (0, 32, True)])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_ragged_shapes(rows, cols, transpose, fmt):
    x = synthetic.student_t((rows, cols), 3, 30.0, seed=rows * 7 + cols)
    sc = np.float32(448.0 / 97.0)
    q, qt, _, am = F.fp8_quantize(x.to(DEV), fmt, scale=torch.tensor([sc], device=DEV),
                                  transpose=transpose, want_amax=True)
    qo, qto = oracle.quantize(bits(x), fmt, sc, transpose=True)
    assert np.array_equal(u8(q), qo)
    if transpose:
        assert np.array_equal(u8(qt), qto)
    assert am.item() == oracle.amax(bits(x))


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 4096, 1000003, 1 << 22])
def test_amax_kernel(n):
    x = synthetic.student_t((n,), 3, 2.0, seed=n)
    a = F.fp8_amax(x.to(DEV))
    assert f32bits(a.cpu().numpy())[0] == f32bits(oracle.amax(bits(x)))


def test_amax_propagates_nan_and_inf():
    x = torch.zeros(10000, dtype=torch.bfloat16)
    x[1234] = float("-inf")
    assert F.fp8_amax(x.to(DEV)).item() == float("inf")
    x[77] = float("nan")
    assert np.isnan(F.fp8_amax(x.to(DEV)).item())


@pytest.mark.parametrize("algo,margin,pow2,fmt,H", [
    (F.AMAX_MAX, 0, False, F.E4M3, 16), (F.AMAX_MAX, 0, True, F.E4M3, 16),
    (F.AMAX_MAX, 1, False, F.E5M2, 16), (F.AMAX_MOST_RECENT, 0, False, F.E4M3, 16),
    (F.AMAX_MAX, 3, True, F.E5M2, 1), (F.AMAX_MAX, 0, False, F.E4M3, 1024),
    (F.AMAX_MAX, 0, False, F.E4M3, 33)])
def test_update_scale_state_machine(algo, margin, pow2, fmt, H):
    rng = np.random.default_rng(H * 10 + margin)
    st = oracle.ScaleState(H)
    hist = torch.zeros(H, dtype=torch.float32, device=DEV)
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = torch.ones(1, dtype=torch.float32, device=DEV)
    sinv = torch.ones(1, dtype=torch.float32, device=DEV)
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    specials = {3: 0.0, 7: float("inf"), 11: float("nan"), 12: 1e-40, 13: 3e38}
    for t in range(2 * H + 5 if H < 100 else 40):
        a = np.float32(abs(rng.standard_normal()) * 10.0 ** rng.integers(-4, 5))
        a = np.float32(specials.get(t, a))
        amax.fill_(float(a))
        F.fp8_update_scale(amax, hist, pos, H, algo, fmt, margin, pow2, scale, sinv)
        oracle.update_scale(st, a, algo, fmt, margin, pow2)
        # status bit 1: the effective amax (the new one, or the history max) is not finite
        nonfinite = (not np.isfinite(a)) if algo == F.AMAX_MOST_RECENT else \
            (not np.all(np.isfinite(st.history)))
        assert F.fp8_device_status(clear=True) == (2 if nonfinite else 0), t
        assert f32bits(scale.cpu().numpy())[0] == f32bits(st.scale)[0], t
        assert f32bits(sinv.cpu().numpy())[0] == f32bits(st.scale_inv)[0], t
        assert pos.item() == st.pos[0]
        assert np.array_equal(f32bits(hist.cpu().numpy()), f32bits(st.history))


def test_update_scale_ring_golden():
    import os
    rows = [list(map(float, l.split())) for l in open(os.path.join(
        os.path.dirname(__file__), "golden", "delayed_scaling_ring.txt")) if l.strip() and l[0] != "#"]
    hist = torch.zeros(16, dtype=torch.float32, device=DEV)
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = torch.ones(1, dtype=torch.float32, device=DEV)
    sinv = torch.ones(1, dtype=torch.float32, device=DEV)
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    for row in rows:
        amax.fill_(row[1])
        F.fp8_update_scale(amax, hist, pos, 16, F.AMAX_MAX, F.E4M3, 0, False, scale, sinv)
        assert scale.item() == row[2]


@pytest.mark.parametrize("gran,shape", [
    (F.GRAN_1x128, (37, 384)), (F.GRAN_1x128, (1, 128)), (F.GRAN_1x128, (1000, 1024)),
    (F.GRAN_128x128, (128, 128)), (F.GRAN_128x128, (384, 640))])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("pow2", [False, True])
def test_block_quantize(gran, shape, fmt, pow2):
    x = synthetic.student_t_rows(shape, 1.0, 3, seed=shape[0] + shape[1])
    x[: min(shape[0], 1), :128] = 0          # an all-zero block
    q, _, sinv, _ = F.fp8_quantize(x.to(DEV), fmt, gran, pow2=pow2)
    qo, so = oracle.block_quantize(bits(x), fmt, 1 if gran == F.GRAN_1x128 else 128, pow2)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(f32bits(sinv.cpu().numpy()), f32bits(so))


@pytest.mark.parametrize("log2n,width", [(20, 4096), (22, 8192), (24, 4096)])
@pytest.mark.parametrize("mag", [1e-2, 1.0, 1e2])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_quantizer_sweep_shapes(log2n, width, mag, fmt):
    """Sweep-shaped tensors: (ii) stale scale 1 with fused amax and transpose
    (saturates at x1e2, underflows at x1e-2); (i) dynamic: amax, scale, cast."""
    rows = (1 << log2n) // width
    x = synthetic.student_t((rows, width), 3, mag, seed=log2n)
    xd = x.to(DEV)
    bx = bits(x)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    q, qt, _, am = F.fp8_quantize(xd, fmt, scale=one, transpose=True, want_amax=True)
    qo, qto = oracle.quantize(bx, fmt, 1.0, transpose=True)
    assert np.array_equal(u8(q), qo) and np.array_equal(u8(qt), qto)
    ao = oracle.amax(bx)
    assert am.item() == ao
    # dynamic: amax pass, scale, cast pass
    amax = F.fp8_amax(xd)
    hist = torch.zeros(1, dtype=torch.float32, device=DEV)
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    sc = torch.ones(1, dtype=torch.float32, device=DEV)
    si = torch.ones(1, dtype=torch.float32, device=DEV)
    F.fp8_update_scale(amax, hist, pos, 1, F.AMAX_MAX, fmt, 0, False, sc, si)
    st = oracle.ScaleState(1)
    oracle.update_scale(st, ao, oracle.ALGO_MAX, fmt)
    assert sc.item() == st.scale[0]
    q2, _, _, _ = F.fp8_quantize(xd, fmt, scale=sc)
    assert np.array_equal(u8(q2), oracle.quantize(bx, fmt, st.scale[0])[0])


@pytest.mark.parametrize("log2n", [28, 30])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_quantizer_full_size_sampled(log2n, fmt):
    """The quantizer sweep's largest tensors, [n/8192 x 8192] t_3 values,
    drawn on the device as the bench draws them: the fused amax bit-exact
    over the whole tensor, and 16 seeded rows of q and 16 of q^T (columns
    of x) bit-exact against the oracle's cast of the same rows and columns,
    with the sweep's stale scale 1 and with the dynamic scale that the
    oracle derives from the amax."""
    width = 8192
    rows = (1 << log2n) // width
    xd = synthetic.student_t((rows, width), 3, 1.0, seed=log2n, device=torch.device(DEV))
    bx = bits(xd.cpu())
    ao = oracle.amax(bx)
    rng = np.random.default_rng(log2n + fmt)
    ri = np.sort(rng.choice(rows, 16, replace=False))
    ci = np.sort(rng.choice(width, 16, replace=False))
    st = oracle.ScaleState(1)
    oracle.update_scale(st, ao, oracle.ALGO_MOST_RECENT, fmt)
    for s in (np.float32(1.0), st.scale[0]):
        sd = torch.tensor([s], dtype=torch.float32, device=DEV)
        q, qt, _, am = F.fp8_quantize(xd, fmt, scale=sd, transpose=True, want_amax=True)
        torch.cuda.synchronize()
        assert f32bits(am.item()) == f32bits(ao)
        assert np.array_equal(u8(q[torch.as_tensor(ri, device=DEV)]), oracle.quantize(bx[ri], fmt, s)[0])
        cols = np.ascontiguousarray(bx[:, ci].T)
        assert np.array_equal(u8(qt[torch.as_tensor(ci, device=DEV)]), oracle.quantize(cols, fmt, s)[0])
        del q, qt
    del xd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("gran", [F.GRAN_1x128, F.GRAN_128x128, F.GRAN_ROW],
                         ids=["dual_1x128", "128x128", "row"])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_recipe_casts_full_size_sampled(gran, fmt):
    """The other recipes' casts with their transposed outputs at the size the
    bench times them (16384 x 7168, per-row heavy-tailed values drawn on the
    device as the bench draws them): seeded sampled rows of q with their
    scales, and sampled rows of q^T (columns of x, whose scales need the
    whole column) with theirs, bit-exact against the oracle's cast of the
    same rows and columns; for 128 x 128 blocks, two sampled 128-row bands."""
    R, C = 16384, 7168
    xd = synthetic.student_t_rows((R, C), 1.0, 3, seed=7, device=torch.device(DEV))
    bx = bits(xd.cpu())
    q, sc, qt, st = F.fp8_quantize_blocks(xd, fmt, gran, transpose=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(gran * 2 + fmt)
    ri = np.sort(rng.choice(R, 16, replace=False))
    ci = np.sort(rng.choice(C, 16, replace=False))
    take = lambda t, idx: t[torch.as_tensor(idx, device=DEV)]
    if gran == F.GRAN_128x128:
        for band in np.sort(rng.choice(R // 128, 2, replace=False)):
            rows = slice(128 * band, 128 * band + 128)
            qo, so = oracle.block_quantize(bx[rows], fmt, 128)
            assert np.array_equal(u8(q[rows]), qo)
            assert np.array_equal(f32bits(sc[band].cpu().numpy()), f32bits(so[0]))
            assert np.array_equal(u8(qt[:, rows]), qo.T)
            assert np.array_equal(f32bits(st[:, band].cpu().numpy()), f32bits(so[0]))
        return
    cast = (lambda a: oracle.block_quantize(a, fmt, 1)) if gran == F.GRAN_1x128 else \
        (lambda a: oracle.row_quantize(a, fmt))
    qo, so = cast(bx[ri])
    assert np.array_equal(u8(take(q, ri)), qo)
    assert np.array_equal(f32bits(take(sc, ri).cpu().numpy()), f32bits(so))
    qto, sto = cast(np.ascontiguousarray(bx[:, ci].T))
    assert np.array_equal(u8(take(qt, ci)), qto)
    assert np.array_equal(f32bits(take(st, ci).cpu().numpy()), f32bits(sto))


@pytest.mark.parametrize("shape", [(128, 128), (384, 256), (1024, 640)])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("pow2", [False, True])
def test_block_1x128_dual_cast(shape, fmt, pow2):
    """One pass gives the 1x128 cast of x and the 1x128 cast of x^T (blocks
    along the columns of x): the wgrad operand layout."""
    x = synthetic.student_t_rows(shape, 1.0, 3, seed=shape[0] * 3 + shape[1])
    x[:128, 128:256] = 0                     # all-zero blocks in both directions
    q, s, qt, st = F.fp8_quantize_blocks(x.to(DEV), fmt, F.GRAN_1x128, pow2=pow2, transpose=True)
    qo, so = oracle.block_quantize(bits(x), fmt, 1, pow2)
    qto, sto = oracle.block_quantize(np.ascontiguousarray(bits(x).T), fmt, 1, pow2)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(f32bits(s.cpu().numpy()), f32bits(so))
    assert np.array_equal(u8(qt), qto)
    assert np.array_equal(f32bits(st.cpu().numpy()), f32bits(sto))


@pytest.mark.parametrize("shape", [(128, 128), (384, 640)])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_block_128x128_cast_with_transpose(shape, fmt):
    x = synthetic.student_t_rows(shape, 0.02, 3, seed=shape[0] + 7)
    q, s, qt, st = F.fp8_quantize_blocks(x.to(DEV), fmt, F.GRAN_128x128, transpose=True)
    qo, so = oracle.block_quantize(bits(x), fmt, 128)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(u8(qt), qo.T)
    assert np.array_equal(f32bits(st.cpu().numpy()), f32bits(so.T))


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("scale", [1.0, 3.0, 1e-3, 2.0 ** 20])
@pytest.mark.parametrize("transpose", [False, True])
def test_cast_counters_every_bf16_pattern(fmt, scale, transpose):
    x = _all_bf16_patterns()
    s = torch.tensor([scale], dtype=torch.float32, device=DEV)
    q, qt, am, counts = F.fp8_quantize_counted(x.to(DEV), fmt, s, transpose=transpose,
                                               want_amax=True)
    qo, _ = oracle.quantize(bits(x), fmt, np.float32(scale))
    assert np.array_equal(u8(q), qo)
    assert tuple(counts.cpu().tolist()) == oracle.cast_counts(bits(x), fmt, scale)
    # the counters accumulate across calls
    F.fp8_quantize_counted(x.to(DEV), fmt, s, counts=counts)
    assert tuple(counts.cpu().tolist()) == tuple(2 * c for c in oracle.cast_counts(bits(x), fmt, scale))


@pytest.mark.parametrize("shape,mag", [((4096, 4096), 1e2), ((4096, 4096), 1e-2), ((37, 61), 30.0),
                                       ((16384, 8192), 1e2), ((16384, 8192), 1e-2)])
def test_cast_counters_sweep_shapes(shape, mag):
    """Stale scale 1 on heavy-tailed data: x1e2 saturates, x1e-2 underflows;
    the last two at the size the bench times the counted cast."""
    x = synthetic.student_t(shape, 3, mag, seed=shape[0] + int(mag))
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    tr = shape[0] % 16 == 0 and shape[1] % 16 == 0
    _, _, _, counts = F.fp8_quantize_counted(x.to(DEV), F.E4M3, one, transpose=tr)
    assert tuple(counts.cpu().tolist()) == oracle.cast_counts(bits(x), F.E4M3, 1.0)


# (4112, 2064): 33 x 17 tiles with ragged edges; (4112, 6144): 33 x 48 tiles,
# enough for the maxima pass to take groups of 4 tiles per CTA, the last
# group of each column ragged
@pytest.mark.parametrize("shape", [(16, 16), (48, 400), (1024, 640), (129, 272), (4112, 2064),
                                   (4112, 6144)])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("pow2", [False, True])
def test_row_cast_and_transposed_column_cast(shape, fmt, pow2):
    x = synthetic.student_t_rows(shape, 1.0, 3, seed=shape[0] * 5 + shape[1])
    x[min(3, shape[0] - 1)] = 0                    # an all-zero row
    x[:, 5] = 0                                    # an all-zero column
    tr = shape[0] % 16 == 0
    q, s, qt, st = F.fp8_quantize_blocks(x.to(DEV), fmt, F.GRAN_ROW, pow2=pow2, transpose=tr)
    qo, so = oracle.row_quantize(bits(x), fmt, pow2)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(f32bits(s.cpu().numpy()), f32bits(so))
    if tr:
        qto, sto = oracle.row_quantize(np.ascontiguousarray(bits(x).T), fmt, pow2)
        assert np.array_equal(u8(qt), qto)
        assert np.array_equal(f32bits(st.cpu().numpy()), f32bits(sto))
