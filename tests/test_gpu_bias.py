"""GPU parity of the bias epilogue and the bias gradient ("Mixed Precision
LLM Training: The Complete Guide", "Transformer Engine internals": te.Linear's
bias) against the oracle.

The bias is added in FP32 before the output rounding, so the forward keeps
the GEMM bound.  The bias gradient is summed in FP32 in a fixed order: per
128-row tile (4 rows per thread, 2 shuffle levels, 8 warps) and then over
the P = ceil(M/128) tiles, a chain of at most 14 + P additions, so
|gpu - sum| <= (16 + P) * 2^-24 * sum|dY| (plus one rounding of an old value
when accumulating).  Two identical calls give identical bits."""
import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import assert_gemm_bound, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    F.build()
    F.lib()
    yield
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0


def _codes(shape, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.randint(0, 0x7C, shape, generator=g, dtype=torch.int32)
    v |= torch.randint(0, 2, shape, generator=g, dtype=torch.int32) << 7
    return v.to(torch.uint8)


def _scales(gran, rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    if gran == F.GRAN_TENSOR:
        shape = (1,)
    elif gran == F.GRAN_ROW:
        shape = (rows,)
    elif gran == F.GRAN_1x128:
        shape = (rows, K // 128)
    else:
        shape = (rows // 128, K // 128)
    return (torch.rand(shape, generator=g) + 0.5) * 2.0 ** -6


@pytest.mark.parametrize("name,M,N,K,ga,gb,out,acc,layout", [
    ("tensor", 128, 384, 256, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_BF16, False, F.LAYOUT_TN),
    ("tensor_ragged", 200, 144, 256, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_BF16, False, F.LAYOUT_TN),
    ("pair", 512, 384, 256, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_BF16, False, F.LAYOUT_TN),
    ("pair_f32_acc", 512, 400, 256, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_F32, True, F.LAYOUT_TN),
    ("row", 512, 384, 256, F.GRAN_ROW, F.GRAN_ROW, F.OUT_BF16, False, F.LAYOUT_TN),
    ("block", 256, 256, 384, F.GRAN_1x128, F.GRAN_128x128, F.OUT_BF16, False, F.LAYOUT_TN),
    # N = 384: the last 256-column tile is half outside the matrix
    ("block_half_tile", 384, 384, 512, F.GRAN_1x128, F.GRAN_128x128, F.OUT_BF16, False,
     F.LAYOUT_TN),
    ("block_colscale_f32", 256, 384, 256, F.GRAN_1x128, F.GRAN_1x128, F.OUT_F32, True, F.LAYOUT_TN),
    ("k0", 64, 96, 0, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_BF16, False, F.LAYOUT_TN),
    ("k0_f32_acc", 64, 96, 0, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_F32, True, F.LAYOUT_TN),
    ("mn_b", 512, 384, 256, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_BF16, False, F.LAYOUT_B_KN),
    ("mn_both_f32_acc", 400, 272, 320, F.GRAN_TENSOR, F.GRAN_TENSOR, F.OUT_F32, True,
     F.LAYOUT_KM_KN),
    ("mn_a_row_small_m", 96, 384, 256, F.GRAN_ROW, F.GRAN_ROW, F.OUT_BF16, False, F.LAYOUT_A_KM),
])
def test_gemm_bias_epilogue(name, M, N, K, ga, gb, out, acc, layout):
    A, B = _codes((M, K), 1), _codes((N, K), 2)
    sa, sb = _scales(ga, M, K, 3), _scales(gb, N, K, 4)
    b = synthetic.normal((N,), 0.5, seed=5)
    prev = None
    D = None
    if out == F.OUT_F32:
        prev = synthetic.normal((M, N), 1.0, seed=6).float()
        D = prev.to(DEV).clone()
    a = A.t().contiguous() if layout & F.LAYOUT_A_KM else A
    b_ = B.t().contiguous() if layout & F.LAYOUT_B_KN else B
    got = F.fp8_gemm(a.to(DEV), F.E4M3, b_.to(DEV), F.E5M2, sa.to(DEV), sb.to(DEV), ga, gb,
                     out=out, D=D, accumulate=acc, bias=b.to(DEV), layout=layout)
    Do, Dabs = oracle.gemm(A.numpy(), F.E4M3, B.numpy(), F.E5M2, sa.numpy(), sb.numpy(), ga, gb,
                           bias=bits(b))
    if prev is not None:
        Do = Do + prev.numpy().astype(np.float64)
    # the bias add is one more fp32 rounding of the output
    assert_gemm_bound(got, Do, Dabs + 2.0 ** -13 * np.abs(Do), prev=prev.numpy() if acc else None,
                      what=name)


def _dbias_tol(dY_bits, M, prev=None):
    _, sabs = oracle.dbias(dY_bits)
    P = (M + 127) // 128
    tol = (16 + P) * 2.0 ** -24 * sabs
    if prev is not None:
        tol = tol + 2.0 ** -23 * (np.abs(prev) + sabs)
    return tol


def _orecipe(r: F.Recipe) -> oracle.Recipe:
    return oracle.Recipe(scaling=r.scaling, margin=r.margin, history_len=r.history_len,
                         algo=r.amax_algo, pow2=bool(r.pow2))


@pytest.mark.parametrize("recipe", [
    F.Recipe(F.SCALING_DELAYED, history_len=16), F.Recipe(F.SCALING_DYNAMIC),
    F.Recipe(F.SCALING_BLOCK), F.Recipe(F.SCALING_ROW)],
    ids=["delayed", "dynamic", "block", "row"])
def test_linear_bias_training_steps(recipe):
    """Three steps with a bias: Y against the oracle's Y + bias, dbias (and
    its accumulation over the steps) against the column sums of dY."""
    M, N, K = 256, 384, 512
    layer = F.Fp8Linear(M, N, K, recipe, device=DEV)
    orec = _orecipe(recipe)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=11)
    b = synthetic.normal((N,), 0.3, seed=12)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    db = torch.zeros(N, dtype=torch.float32, device=DEV)
    db_o = np.zeros(N)
    for step in range(3):
        X = synthetic.with_outlier_channels((M, K), 1.0, 4, 50.0, seed=20 + step)
        dY = synthetic.student_t((M, N), 3, 1e-3, seed=30 + step)
        acc = step > 0
        Y = layer.forward(X.to(DEV), W.to(DEV), bias=b.to(DEV))
        prev_db = db.cpu().numpy().astype(np.float64)
        layer.backward(dY.to(DEV), dW=dW, accumulate_dW=acc, dbias=db)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost, bias=bits(b))
        oracle.linear_bwd(bits(dY), orec, ost)
        assert_gemm_bound(Y, Yo, Yabs + 2.0 ** -13 * np.abs(Yo), what=f"Y step {step}")
        s, _ = oracle.dbias(bits(dY))
        want = s + (prev_db if acc else 0.0)
        tol = _dbias_tol(bits(dY), M, prev_db if acc else None)
        err = np.abs(db.cpu().numpy().astype(np.float64) - want)
        assert np.all(err <= tol), f"step {step}: max err/tol {np.max(err / tol)}"


@pytest.mark.parametrize("M,N", [(144, 256), (8192, 12288)])
def test_dbias_is_deterministic_and_within_bound(M, N):
    """dY of the Llama-2-7B QKV linear (8192 x 12288), and a token count that
    is not a multiple of 128: two backward calls give identical bits."""
    K = 256
    rec = F.Recipe(F.SCALING_DELAYED, history_len=16)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    X = synthetic.normal((M, K), 1.0, seed=40).to(DEV)
    W = synthetic.normal((N, K), 0.02, seed=41).to(DEV)
    dY = synthetic.student_t((M, N), 3, 1e-3, seed=42)
    out = []
    for _ in range(2):
        layer.forward(X, W)
        db = torch.empty(N, dtype=torch.float32, device=DEV)
        layer.backward(dY.to(DEV), dbias=db)
        out.append(db.cpu())
    assert torch.equal(out[0].view(torch.int32), out[1].view(torch.int32))
    s, _ = oracle.dbias(bits(dY))
    err = np.abs(out[0].numpy().astype(np.float64) - s)
    assert np.all(err <= _dbias_tol(bits(dY), M))
