"""The bounded-wait timeout path, made to run without any GPU fault: a test
hook shortens the single-CTA GEMM kernel's epilogue wait for a full
accumulator (a wait with no asynchronous work of its own behind it) so that it
gives up on a long GEMM.  The kernel must return with bit 0 of the device
status word set, the context must stay usable, and the next call with the
normal limit must be correct."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import assert_gemm_bound, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEFAULT_NS = 2_000_000_000


def _hook():
    F.build()
    fn = F.lib().fp8_test_set_epilogue_wait_ns
    fn.argtypes = [ctypes.c_uint64]
    fn.restype = ctypes.c_int
    return fn


def _codes(r, c, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    v = torch.randint(0, 0x7C, (r, c), generator=g, device=DEV, dtype=torch.int32)
    v |= torch.randint(0, 2, (r, c), generator=g, device=DEV, dtype=torch.int32) << 7
    return v.to(torch.uint8)


@pytest.fixture()
def short_epilogue_wait():
    fn = _hook()
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0
    assert fn(1000) == 0          # 1 us: far below one 128 x 256 tile of K = 131072
    try:
        yield
    finally:
        torch.cuda.synchronize()
        assert fn(DEFAULT_NS) == 0
        F.fp8_device_status()     # leave the word clear for the next test


def test_epilogue_wait_runs_out_then_the_next_gemm_is_correct(short_epilogue_wait):
    M, N, K = 128, 256, 131072     # one tile on the single-CTA kernel (M < 256)
    A, B = _codes(M, K, 1), _codes(N, K, 2)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    D = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    # the call itself succeeds; the kernel reports the timeout through the
    # status word, which the host reads after synchronising
    F.fp8_gemm(A, F.E4M3, B, F.E4M3, one, one, out=F.OUT_F32, D=D)
    assert F.fp8_device_status(clear=False) & F.STATUS_TIMEOUT
    with pytest.raises(F.Fp8Error) as e:
        F.check_device_status()
    assert e.value.status == -5
    assert F.fp8_device_status() == 0          # read and cleared
    assert _hook()(DEFAULT_NS) == 0
    D2 = F.fp8_gemm(A, F.E4M3, B, F.E4M3, one, one, out=F.OUT_F32)
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0
    Do, Dabs = oracle.gemm(u8(A), F.E4M3, u8(B), F.E4M3, np.float32([1.0]), np.float32([1.0]))
    assert_gemm_bound(D2, Do, Dabs, what="GEMM after the timeout")


def test_layer_with_check_status_raises_on_timeout(short_epilogue_wait):
    """Fp8Linear(check_status=True) turns the status word into an exception
    after the forward whose GEMM gave up."""
    M, N, K = 128, 256, 131072
    layer = F.Fp8Linear(M, N, K, F.Recipe(F.SCALING_DYNAMIC), device=DEV, check_status=True)
    X = synthetic.normal((M, K), 1.0, seed=3, device=DEV)
    W = synthetic.normal((N, K), 0.02, seed=4, device=DEV)
    with pytest.raises(F.Fp8Error) as e:
        layer.forward(X, W)
    assert e.value.status == -5
    assert _hook()(DEFAULT_NS) == 0
    layer.forward(X, W)                         # the normal limit: no exception
    dY = synthetic.normal((M, N), 1e-3, seed=5, device=DEV)
    layer.backward(dY)
