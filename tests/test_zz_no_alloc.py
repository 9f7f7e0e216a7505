"""fp8_linear_bwd_noalloc -- the backward entry point for callers that cannot
allocate device memory (its scratch is a fixed device array inside the
library) -- against the existing fp8_linear_bwd with a caller workspace, on
two calls in a row.  Called through the C ABI with ctypes.  This file sorts
last so that a run stopping at the first failure has run every other test
first; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import assert_gemm_bound, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc():
    F.build()
    L = F.lib()
    fn = L.fp8_linear_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                   ctypes.POINTER(F.Recipe), ctypes.POINTER(F.LinearStateC), ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _same_bits(got, want, what):
    """dX (bf16) and dW (fp32) of the two entry points: the same kernels on
    the same codes, so the same bits."""
    ib = torch.int16 if got.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(got.view(ib), want.view(ib)), what


def test_noalloc_backward_matches_workspace_backward():
    """Delayed scaling over two calls with dW accumulated: the same bits as
    fp8_linear_bwd with a workspace, and both within the GEMM bound of the
    oracle."""
    fn = _noalloc()
    M, N, K = 512, 768, 1024
    rec = F.Recipe(F.SCALING_DELAYED, history_len=16)
    ref_layer = F.Fp8Linear(M, N, K, rec, device=DEV)    # fp8_linear_bwd + workspace
    na_layer = F.Fp8Linear(M, N, K, rec, device=DEV)     # fp8_linear_bwd_noalloc
    orec = oracle.Recipe(scaling=oracle.SCALING_DELAYED, history_len=16)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=7)
    dW_ref = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    dW_na = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        X = synthetic.with_outlier_channels((M, K), 1.0, 4, 50.0, seed=10 + step)
        dY = synthetic.normal((M, N), 1e-3, seed=20 + step)
        ref_layer.forward(X.to(DEV), W.to(DEV))
        na_layer.forward(X.to(DEV), W.to(DEV))
        dX_ref, _ = ref_layer.backward(dY.to(DEV), dW=dW_ref, accumulate_dW=step > 0)
        dX_na = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
        dYd = dY.to(DEV)
        st = fn(dYd.data_ptr(), M, N, K, ctypes.byref(rec), ctypes.byref(na_layer.c_state),
                dX_na.data_ptr(), dW_na.data_ptr(), int(step > 0), stream)
        assert st == 0, F.fp8_last_error()
        torch.cuda.synchronize()
        _same_bits(dX_na, dX_ref, f"dX call {step}")
        _same_bits(dW_na, dW_ref, f"dW call {step}")
        # tolerance of the GEMM tests: 2e-3 * sum|a b| * s_a * s_b (+ bf16 rounding)
        oracle.linear_fwd(bits(X), bits(W), orec, ost)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost)
        assert_gemm_bound(dX_na, dXo, dXabs, what=f"dX call {step}")
        if step == 0:
            assert_gemm_bound(dW_na, dWo, dWabs, what="dW call 0")
        assert torch.equal(na_layer.scale, ref_layer.scale)
        assert torch.equal(na_layer.history, ref_layer.history)
    assert F.fp8_device_status() == 0


@pytest.mark.parametrize("mode,transposes", [
    (F.SCALING_DELAYED, True),     # dY_q and dY_q^T: 2*M*N bytes of scratch
    (F.SCALING_BLOCK, False),      # 1x128 dY and dY^T codes plus their scale arrays
    (F.SCALING_ROW, False),        # per-token dY and per-channel dY^T plus their scales
], ids=["delayed_transposed_copies", "block", "per_row"])
def test_noalloc_matches_workspace_in_every_scratch_layout(mode, transposes):
    """The recipes whose backward puts two dY operands (and scale arrays) in
    the scratch: two calls in a row with dW accumulated, bit for bit the
    workspace backward's results."""
    fn = _noalloc()
    M, N, K = 512, 768, 1024
    rec = F.Recipe(mode, history_len=16)
    ref_layer = F.Fp8Linear(M, N, K, rec, device=DEV, transposes=transposes)
    na_layer = F.Fp8Linear(M, N, K, rec, device=DEV, transposes=transposes)
    W = synthetic.student_t_rows((N, K), 0.02, 3, seed=8, device=DEV)
    dW_ref = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    dW_na = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        X = synthetic.student_t_rows((M, K), 1.0, 3, seed=30 + step, device=DEV)
        dY = synthetic.normal((M, N), 1e-3, seed=40 + step, device=DEV)
        ref_layer.forward(X, W)
        na_layer.forward(X, W)
        dX_ref, _ = ref_layer.backward(dY, dW=dW_ref, accumulate_dW=step > 0)
        dX_na = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
        st = fn(dY.data_ptr(), M, N, K, ctypes.byref(rec), ctypes.byref(na_layer.c_state),
                dX_na.data_ptr(), dW_na.data_ptr(), int(step > 0), stream)
        assert st == 0, F.fp8_last_error()
        torch.cuda.synchronize()
        _same_bits(dX_na, dX_ref, f"dX call {step}")
        _same_bits(dW_na, dW_ref, f"dW call {step}")
    assert F.fp8_device_status() == 0


def test_noalloc_rejects_shapes_beyond_the_scratch():
    fn = _noalloc()
    rec = F.Recipe(F.SCALING_DELAYED, history_len=16)
    fake = 0x10000   # 16-byte aligned, never dereferenced: the calls fail validation
    p = ctypes.c_void_p(fake)
    # a state whose arrays are all set, without transposed copies: the
    # scratch holds dY_q alone, and 8192 * 8192 bytes > 32 MiB is rejected
    # before any device work
    st = F.LinearStateC(*([fake] * len(F.LinearStateC._fields_)))
    st.x_qt = st.w_qt = None
    assert fn(p, 8192, 8192, 4096, ctypes.byref(rec), ctypes.byref(st), p, p, 0, None) == -2
    assert "scratch" in F.fp8_last_error()
    # with them it also holds dY_q^T: 2 * 8192 * 4096 bytes > 32 MiB
    st_t = F.LinearStateC(*([fake] * len(F.LinearStateC._fields_)))
    assert fn(p, 8192, 4096, 4096, ctypes.byref(rec), ctypes.byref(st_t), p, p, 0, None) == -2
    assert "scratch" in F.fp8_last_error()


def test_noalloc_takes_twice_the_tokens_without_transposed_copies():
    """8192 x 4096 (32 MiB of dY codes): beyond the scratch with transposed
    copies, within it when the backward reads the codes MN-major; the result
    equals the workspace backward's."""
    fn = _noalloc()
    M, N, K = 8192, 4096, 512
    rec = F.Recipe(F.SCALING_DYNAMIC)
    ref_layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    na_layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    X = synthetic.normal((M, K), 1.0, seed=3, device=DEV)
    W = synthetic.normal((N, K), 0.02, seed=4, device=DEV)
    dY = synthetic.normal((M, N), 1e-3, seed=5, device=DEV)
    ref_layer.forward(X, W)
    na_layer.forward(X, W)
    dX_ref, dW_ref = ref_layer.backward(dY)
    dX_na = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    dW_na = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    st = fn(dY.data_ptr(), M, N, K, ctypes.byref(rec), ctypes.byref(na_layer.c_state),
            dX_na.data_ptr(), dW_na.data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0, F.fp8_last_error()
    torch.cuda.synchronize()
    _same_bits(dX_na, dX_ref, "dX")
    _same_bits(dW_na, dW_ref, "dW")
    assert torch.equal(na_layer.scale, ref_layer.scale)


def _scratch_addresses():
    """(address from the per-context table, fresh lookup) in the current context."""
    fn = F.lib().fp8_test_noalloc_scratch
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p)]
    fn.restype = ctypes.c_int
    cached, fresh = ctypes.c_void_p(), ctypes.c_void_p()
    assert fn(ctypes.byref(cached), ctypes.byref(fresh)) == 0, F.fp8_last_error()
    return cached.value, fresh.value


def test_noalloc_scratch_address_belongs_to_the_current_context():
    """The scratch address is looked up once per CUDA context: in the primary
    context and in a second context of the same device (made current with the
    driver API) it equals a fresh lookup, and the primary context's entry is
    still right after the other context has been used."""
    F.build()
    torch.zeros(1, device=DEV)
    torch.cuda.synchronize()
    c0, f0 = _scratch_addresses()
    assert c0 and c0 == f0
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        create, pop, destroy = cu.cuCtxCreate_v2, cu.cuCtxPopCurrent_v2, cu.cuCtxDestroy_v2
    except (OSError, AttributeError):
        pytest.skip("the driver API's context calls are not available")
    create.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint, ctypes.c_int]
    pop.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    destroy.argtypes = [ctypes.c_void_p]
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    ctx = ctypes.c_void_p()
    assert create(ctypes.byref(ctx), 0, dev.value) == 0
    try:
        c1, f1 = _scratch_addresses()
        assert c1 and c1 == f1
    finally:
        popped = ctypes.c_void_p()
        assert pop(ctypes.byref(popped)) == 0 and popped.value == ctx.value
        assert destroy(ctx) == 0
    c2, f2 = _scratch_addresses()
    assert c2 == f2 == c0
