"""GPU parity of the stochastic-rounding cast ("Mixed Precision LLM
Training: The Complete Guide", "Stochastic rounding") against the CPU oracle:
every code and amax bit-exact, for both FP8 formats, flat and transposed
launches, ragged shapes, 64-bit seeds and offsets, special values and the
full-size gradient tensor of the Llama-2-7B linears."""
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


def _check(x, fmt, scale, seed, offset, transpose):
    s = torch.tensor([scale], dtype=torch.float32, device=DEV)
    q, qt, am = F.fp8_quantize_sr(x.to(DEV), fmt, s, seed, offset, transpose=transpose,
                                  want_amax=True)
    qo, qto = oracle.quantize_sr(bits(x), fmt, np.float32(scale), seed, offset, transpose=True)
    got = u8(q)
    bad = np.argwhere(got != qo)
    assert bad.size == 0, (f"{len(bad)} of {qo.size} codes differ, first at {tuple(bad[0])}: "
                           f"gpu {got[tuple(bad[0])]:#04x} oracle {qo[tuple(bad[0])]:#04x}")
    if transpose:
        assert np.array_equal(u8(qt), qto)
    if x.numel():
        assert f32bits(am.cpu().numpy())[0] == f32bits(oracle.amax(bits(x)))


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
@pytest.mark.parametrize("scale", [1.0, 448.0 / 3.0, 1e-3, 2.0 ** 20, 1.2e-38])
@pytest.mark.parametrize("transpose", [False, True])
def test_every_bf16_pattern(fmt, scale, transpose):
    x = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(256, 256)
    _check(x, fmt, scale, seed=0x5EED, offset=3, transpose=transpose)


@pytest.mark.parametrize("rows,cols,transpose", [
    (1, 1, False), (3, 37, False), (1, 15, False), (17, 16, False), (129, 1000, False),
    (16, 16, True), (144, 400, True), (1040, 2064, True), (0, 64, False), (0, 32, True)])
@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2])
def test_ragged_shapes(rows, cols, transpose, fmt):
    x = synthetic.student_t((rows, cols), 3, 30.0, seed=rows * 7 + cols)
    _check(x, fmt, 448.0 / 97.0, seed=rows + 1, offset=cols, transpose=transpose)


@pytest.mark.parametrize("seed,offset", [(0, 0), (0xFFFFFFFFFFFFFFFF, 0xFFFFFFFFFFFFFFFF),
                                         (0xDEADBEEF12345678, (1 << 40) + 5)])
def test_64bit_seed_and_offset(seed, offset):
    x = synthetic.normal((256, 512), 0.02, seed=5)
    _check(x, F.E5M2, 2.0 ** 14, seed, offset, transpose=True)
    _check(x, F.E5M2, 2.0 ** 14, seed, offset, transpose=False)


def test_full_size_gradient_tensor():
    """dY of the Llama-2-7B linears (8192 tokens x 4096 features), E5M2 with
    the scale a delayed recipe would set, cast and transposed in one pass."""
    x = synthetic.normal((8192, 4096), 1e-4, seed=21)
    scale = float(np.float32(57344.0 / float(x.float().abs().max())))
    _check(x, F.E5M2, scale, seed=2024, offset=17, transpose=True)
    _check(x, F.E5M2, scale, seed=2024, offset=17, transpose=False)


def test_gpu_draws_are_unbiased():
    """Mean of the decoded codes of a constant tensor: within 5 sigma of the
    scaled value (round to nearest is far off it)."""
    x = torch.full((2048, 2048), 0.3, dtype=torch.bfloat16, device=DEV)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    q, _, _ = F.fp8_quantize_sr(x, F.E4M3, one, seed=77, offset=0)
    d = q.view(torch.float8_e4m3fn).float().double()
    v = float(x[0, 0].float())
    lo, hi = 0.28125, 0.3125
    f = (v - lo) / (hi - lo)
    sigma = (hi - lo) * (f * (1 - f) / d.numel()) ** 0.5
    assert abs(d.mean().item() - v) < 5 * sigma


@pytest.mark.parametrize("scaling", [F.SCALING_DELAYED, F.SCALING_DYNAMIC], ids=["delayed", "dynamic"])
def test_linear_with_stochastic_gradient_cast(scaling):
    """recipe.sr_grad through fp8_linear_bwd: the dY codes bit-exact with the
    oracle's quantize_sr(seed, call number) at every step, the scaling state
    bit-exact, dX / dW within the GEMM bound, dbias unaffected, and the
    device counter advanced once per call."""
    from tests.helpers import assert_gemm_bound
    M, N, K = 256, 384, 512
    seed = 0xC0FFEE12345
    rec = F.Recipe(scaling, history_len=16, sr_grad=True)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV, sr_seed=seed)
    orec = oracle.Recipe(scaling=scaling, history_len=16, sr_grad=True)
    ost = oracle.LinearState(orec, sr_seed=seed)
    W = synthetic.normal((N, K), 0.02, seed=3)
    db = torch.zeros(N, dtype=torch.float32, device=DEV)
    for step in range(5):
        X = synthetic.with_outlier_channels((M, K), 1.0, 4, 50.0, seed=10 + step)
        dY = synthetic.student_t((M, N), 3, 1e-3, seed=20 + step)
        layer.forward(X.to(DEV), W.to(DEV))
        dX, dW = layer.backward(dY.to(DEV), dbias=db)
        oracle.linear_fwd(bits(X), bits(W), orec, ost)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost)
        assert np.array_equal(u8(layer.workspace[:M * N].view(M, N)), ost.dy_q), step
        for r in range(3):
            assert f32bits(layer.scale[r].cpu().numpy()) == f32bits(ost.roles[r].scale[0])
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, what=f"dW step {step}")
        s, sabs = oracle.dbias(bits(dY))
        assert np.all(np.abs(db.cpu().numpy() - s) <= (18 * 2.0 ** -24) * sabs)
    key = layer.sr_key.cpu().numpy().view(np.uint64)
    assert int(key[0]) == seed and int(key[1]) == 5
