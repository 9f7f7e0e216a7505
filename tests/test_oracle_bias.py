"""Pins of the oracle's bias and bias gradient.

"Mixed Precision LLM Training: The Complete Guide", "Transformer Engine
internals": te.Linear carries a bias, added to every row of X . W^T; its
gradient is therefore the sum of dY over the rows (tokens).  Pinned against
closed forms, exact rational arithmetic on a tiny case, and PyTorch's own
linear and autograd in fp64 -- not against a re-typing of the oracle.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
import synthetic
from oracle import E4M3
from tests.helpers import bits


def _bf16_bits(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def test_zero_operand_gives_the_bias_exactly():
    rng = np.random.default_rng(0)
    A = np.zeros((32, 64), np.uint8)
    B = rng.integers(0, 0x7F, (48, 64)).astype(np.uint8)
    b = _bf16_bits(torch.from_numpy(rng.standard_normal(48).astype(np.float32)))
    D, _ = oracle.gemm(A, E4M3, B, E4M3, 0.5, 3.0, bias=b)
    want = oracle.bf16_to_f32(b).astype(np.float64)
    assert np.array_equal(D, np.broadcast_to(want, D.shape))


def test_linear_forward_with_bias_matches_torch_linear():
    X = synthetic.normal((64, 128), 1.0, seed=1)
    W = synthetic.normal((96, 128), 0.02, seed=2)
    b = synthetic.normal((96,), 0.1, seed=3)
    rec = oracle.Recipe(scaling=oracle.SCALING_DYNAMIC)
    st = oracle.LinearState(rec)
    Y, _ = oracle.linear_fwd(bits(X), bits(W), rec, st, bias=bits(b))
    # the same quantised operands, dequantised, through torch's linear in fp64
    xq = torch.from_numpy(oracle.decode(st.x_q.ravel(), E4M3).reshape(st.x_q.shape))
    wq = torch.from_numpy(oracle.decode(st.w_q.ravel(), E4M3).reshape(st.w_q.shape))
    sx, sw = st.sinv_fwd
    ref = torch.nn.functional.linear(xq * float(np.ravel(sx)[0]), wq * float(np.ravel(sw)[0]),
                                     b.double())
    assert np.allclose(Y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_bias_gradient_matches_autograd():
    M, N, K = 200, 48, 32
    dY = synthetic.student_t((M, N), 3, 1e-3, seed=4)
    x = torch.randn(M, K, dtype=torch.float64)
    w = torch.randn(N, K, dtype=torch.float64)
    bvec = torch.zeros(N, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.linear(x, w, bvec)
    y.backward(dY.double())
    got, gabs = oracle.dbias(bits(dY))
    assert np.allclose(got, bvec.grad.numpy(), rtol=1e-12, atol=1e-18)
    assert np.all(gabs >= np.abs(got))


def test_bias_gradient_closed_form_and_exact_sum():
    # identical rows: the sum is M times the row, exactly
    row = synthetic.normal((1, 40), 1.0, seed=5)
    dY = row.repeat(300, 1)
    got, _ = oracle.dbias(bits(dY))
    assert np.array_equal(got, 300.0 * row.double().numpy()[0])
    # a tiny case summed in exact rationals
    dY = synthetic.student_t((7, 5), 3, 10.0, seed=6)
    vals = dY.float().numpy()
    exact = [sum(Fraction(float(vals[m, n])) for m in range(7)) for n in range(5)]
    got, _ = oracle.dbias(bits(dY))
    assert [Fraction(float(g)) for g in got] == exact
