"""Scaled FP8 linear layer for NVIDIA GB300 (sm_103a).

A thin Python binding of the C-ABI library ``libfp8linear.so`` (declared in
``include/fp8linear.h``).  The functions here carry the C names and only
marshal arguments: torch tensors supply device memory and the current CUDA
stream, and every step of the computation runs in the library's kernels.
There is no fallback: if the library has not been built (``build()``), or
no GPU is present, every call raises.

The method is the FP8 linear layer of "Mixed Precision LLM Training: The
Complete Guide": E4M3 forward operands, E5M2 gradients, FP32 accumulation,
per-tensor (dynamic or delayed/history) or block-wise (1x128 / 128x128)
scales.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "E4M3", "E5M2", "OUT_BF16", "OUT_F32", "AMAX_MAX", "AMAX_MOST_RECENT",
    "GRAN_TENSOR", "GRAN_1x128", "GRAN_128x128", "GRAN_ROW", "SCALE_POW2", "LAYOUT_TN", "LAYOUT_B_KN", "LAYOUT_A_KM", "LAYOUT_KM_KN",
    "SCALING_DELAYED", "SCALING_DYNAMIC", "SCALING_BLOCK", "SCALING_ROW",
    "Fp8Error", "Recipe", "LinearStateC", "Fp8Linear", "build", "lib", "library_path",
    "fp8_amax", "fp8_update_scale", "fp8_quantize", "fp8_quantize_blocks",
    "fp8_quantize_counted", "fp8_quantize_sr", "fp8_gemm", "fp8_gemm_group", "GemmArgsC",
    "fp8_workspace_size",
    "fp8_linear_fwd", "fp8_linear_bwd", "fp8_last_error", "fp8_device_status",
    "check_device_status", "Fp8NumericsError", "STATUS_TIMEOUT", "STATUS_NONFINITE",
]

E4M3, E5M2 = 0, 1
OUT_BF16, OUT_F32 = 0, 1
AMAX_MAX, AMAX_MOST_RECENT = 0, 1
GRAN_TENSOR, GRAN_1x128, GRAN_128x128, GRAN_ROW = 0, 1, 2, 3
SCALE_POW2 = 16   # OR'd into a block granularity: every factor is a power of two
LAYOUT_TN = 0
LAYOUT_B_KN = 1       # B stored [K, N]
LAYOUT_A_KM = 2       # A stored [K, M]
LAYOUT_KM_KN = 3      # both
SCALING_DELAYED, SCALING_DYNAMIC, SCALING_BLOCK, SCALING_ROW = 0, 1, 2, 3

_STATUS = {0: "FP8_OK", -1: "FP8_ERR_INVALID_ARG", -2: "FP8_ERR_SHAPE", -3: "FP8_ERR_ALIGN",
           -4: "FP8_ERR_CUDA", -5: "FP8_ERR_TIMEOUT", -6: "FP8_ERR_UNSUPPORTED"}

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libfp8linear.so")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import nvcc_build
    return nvcc_build.build(force=force)


class Fp8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class Recipe(ctypes.Structure):
    """fp8_recipe_t: HYBRID recipe (E4M3 forward, E5M2 backward) by default."""
    _fields_ = [("scaling", ctypes.c_int32), ("margin", ctypes.c_int32),
                ("history_len", ctypes.c_int32), ("amax_algo", ctypes.c_int32),
                ("pow2", ctypes.c_int32), ("fwd_format", ctypes.c_int32),
                ("bwd_format", ctypes.c_int32), ("sr_grad", ctypes.c_int32)]

    def __init__(self, scaling=SCALING_DELAYED, margin=0, history_len=16, amax_algo=AMAX_MAX,
                 pow2=False, fwd_format=E4M3, bwd_format=E5M2, sr_grad=False):
        super().__init__(scaling, margin, history_len, amax_algo, int(bool(pow2)), fwd_format,
                         bwd_format, int(bool(sr_grad)))


_vp = ctypes.c_void_p


class GemmArgsC(ctypes.Structure):
    """fp8_gemm_args_t: the arguments of one fp8_gemm call."""
    _fields_ = [("A", _vp), ("fa", ctypes.c_int32), ("B", _vp), ("fb", ctypes.c_int32),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("ga", ctypes.c_int32), ("scale_inv_a", _vp),
                ("gb", ctypes.c_int32), ("scale_inv_b", _vp), ("bias", _vp), ("D", _vp),
                ("out", ctypes.c_int32), ("accumulate", ctypes.c_int32)]


class LinearStateC(ctypes.Structure):
    """fp8_linear_state_t: device pointers of one layer's scaling state."""
    _fields_ = [("scale", _vp), ("scale_inv", _vp), ("amax", _vp), ("history", _vp),
                ("pos", _vp), ("x_q", _vp), ("x_qt", _vp), ("w_q", _vp), ("w_qt", _vp),
                ("x_sinv", _vp), ("w_sinv", _vp), ("qscale_inv", _vp), ("x_sinv_t", _vp),
                ("w_sinv_t", _vp), ("sr_key", _vp)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfp8linear.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(scaled_fp8_linear_gb300.build())")
    L = ctypes.CDLL(path)
    i, i64, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.fp8_amax.argtypes = [_vp, i64, _vp, _vp]
    L.fp8_update_scale.argtypes = [_vp, _vp, _vp, i, i, i, i, i, _vp, _vp, _vp]
    L.fp8_quantize.argtypes = [_vp, i64, i64, i, i, _vp, i, _vp, _vp, _vp, _vp, _vp, _vp]
    L.fp8_quantize_counted.argtypes = [_vp, i64, i64, i, _vp, _vp, _vp, _vp, _vp, _vp]
    L.fp8_quantize_sr.argtypes = [_vp, i64, i64, i, _vp, ctypes.c_uint64, ctypes.c_uint64,
                                  _vp, _vp, _vp, _vp]
    L.fp8_gemm.argtypes = [_vp, i, _vp, i, i64, i64, i64, i, i, _vp, i, _vp, _vp, _vp, i, i, _vp]
    L.fp8_gemm_group.argtypes = [ctypes.POINTER(GemmArgsC), ctypes.POINTER(GemmArgsC), _vp]
    L.fp8_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(Recipe)]
    L.fp8_workspace_size.restype = sz
    L.fp8_linear_fwd.argtypes = [_vp, _vp, _vp, i64, i64, i64, ctypes.POINTER(Recipe),
                                 ctypes.POINTER(LinearStateC), _vp, _vp, sz, _vp]
    L.fp8_linear_bwd.argtypes = [_vp, i64, i64, i64, ctypes.POINTER(Recipe),
                                 ctypes.POINTER(LinearStateC), _vp, _vp, i, _vp, _vp, sz, _vp]
    L.fp8_last_error.restype = ctypes.c_char_p
    L.fp8_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i]
    for name in ("fp8_amax", "fp8_update_scale", "fp8_quantize", "fp8_quantize_counted",
                 "fp8_quantize_sr", "fp8_gemm", "fp8_gemm_group", "fp8_linear_fwd",
                 "fp8_linear_bwd", "fp8_device_status"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def fp8_last_error() -> str:
    return lib().fp8_last_error().decode()


class Fp8NumericsError(RuntimeError):
    """A scale update met a non-finite amax (a NaN or Inf in a cast tensor,
    or still in its amax history) and kept the previous scale."""


def _check(status: int) -> None:
    if status != 0:
        raise Fp8Error(status, fp8_last_error())


# The current stream's handle without building a torch.cuda.Stream object
# (about 0.1 us against 3 us a call); the public call where it is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, what, dtype=None, device=True):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a tensor")
    if device and not t.is_cuda:
        raise ValueError(f"{what}: must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{what}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    return t.data_ptr()


_U8 = (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)


# ------------------------------------------------------------------ raw calls

def fp8_amax(x: torch.Tensor, amax: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """max |x| of a bf16 tensor into a 1-element fp32 device tensor."""
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().fp8_amax(_ptr(x, "x", torch.bfloat16), x.numel(),
                          _ptr(amax, "amax", torch.float32), _stream(stream)))
    return amax


def fp8_update_scale(amax, history, pos, history_len, algo, fmt, margin, pow2, scale,
                     scale_inv, stream=None) -> None:
    """One scale-update step on device state (see include/fp8linear.h)."""
    _check(lib().fp8_update_scale(
        _ptr(amax, "amax", torch.float32), _ptr(history, "history", torch.float32),
        _ptr(pos, "pos", torch.int32), int(history_len), int(algo), int(fmt), int(margin),
        int(bool(pow2)), _ptr(scale, "scale", torch.float32),
        _ptr(scale_inv, "scale_inv", torch.float32), _stream(stream)))


def _scale_shape(gran, rows, cols):
    if gran == GRAN_ROW:
        return (rows,)
    return (rows // (1 if gran == GRAN_1x128 else 128), cols // 128)


def _scale_shape_t(gran, rows, cols):
    if gran == GRAN_ROW:
        return (cols,)
    return (cols, rows // 128) if gran == GRAN_1x128 else (cols // 128, rows // 128)


def fp8_quantize(x: torch.Tensor, fmt: int, granularity: int = GRAN_TENSOR, scale=None,
                 pow2: bool = False, q=None, q_t=None, transpose: bool = False,
                 scale_inv_blocks=None, amax_out=None, want_amax: bool = False,
                 scale_inv_blocks_t=None, stream=None):
    """Cast a 2-D bf16 tensor to FP8 codes (uint8).  Returns
    (q, q_t or None, scale_inv_blocks or None, amax or None); in block modes
    with transpose=True the transposed block scales are in
    `scale_inv_blocks_t` (allocated here if not given) -- see
    fp8_quantize_blocks for a call that returns them."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
    if transpose and q_t is None:
        q_t = torch.empty(cols, rows, dtype=torch.uint8, device=dev)
    if granularity != GRAN_TENSOR and scale_inv_blocks is None:
        scale_inv_blocks = torch.empty(*_scale_shape(granularity, rows, cols), dtype=torch.float32,
                                       device=dev)
    if granularity != GRAN_TENSOR and q_t is not None and scale_inv_blocks_t is None:
        scale_inv_blocks_t = torch.empty(*_scale_shape_t(granularity, rows, cols),
                                         dtype=torch.float32, device=dev)
    if want_amax and amax_out is None:
        amax_out = torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().fp8_quantize(
        _ptr(x, "x", torch.bfloat16), rows, cols, int(fmt), int(granularity),
        _ptr(scale, "scale", torch.float32), int(bool(pow2)), _ptr(q, "q", _U8),
        _ptr(q_t, "q_t", _U8), _ptr(scale_inv_blocks, "scale_inv_blocks", torch.float32),
        _ptr(scale_inv_blocks_t, "scale_inv_blocks_t", torch.float32),
        _ptr(amax_out, "amax_out", torch.float32), _stream(stream)))
    return q, q_t, scale_inv_blocks, amax_out


def fp8_quantize_counted(x: torch.Tensor, fmt: int, scale, counts=None, q=None, q_t=None,
                         transpose: bool = False, amax_out=None, want_amax: bool = False,
                         stream=None):
    """Per-tensor cast with fused dashboard counters.  Returns
    (q, q_t or None, amax or None, counts) where counts is a 2-element int64
    device tensor [underflow, saturated] that the call adds to."""
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
    if transpose and q_t is None:
        q_t = torch.empty(cols, rows, dtype=torch.uint8, device=dev)
    if want_amax and amax_out is None:
        amax_out = torch.empty(1, dtype=torch.float32, device=dev)
    if counts is None:
        counts = torch.zeros(2, dtype=torch.int64, device=dev)
    _check(lib().fp8_quantize_counted(
        _ptr(x, "x", torch.bfloat16), rows, cols, int(fmt), _ptr(scale, "scale", torch.float32),
        _ptr(q, "q", _U8), _ptr(q_t, "q_t", _U8), _ptr(amax_out, "amax_out", torch.float32),
        _ptr(counts, "counts", torch.int64), _stream(stream)))
    return q, q_t, amax_out, counts


def fp8_quantize_sr(x: torch.Tensor, fmt: int, scale, seed: int, offset: int = 0, q=None,
                    q_t=None, transpose: bool = False, amax_out=None, want_amax: bool = False,
                    stream=None):
    """Per-tensor cast with stochastic rounding (Philox-4x32-10 keyed by seed,
    counter offset).  Returns (q, q_t or None, amax or None)."""
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
    if transpose and q_t is None:
        q_t = torch.empty(cols, rows, dtype=torch.uint8, device=dev)
    if want_amax and amax_out is None:
        amax_out = torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().fp8_quantize_sr(
        _ptr(x, "x", torch.bfloat16), rows, cols, int(fmt), _ptr(scale, "scale", torch.float32),
        int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFFFFFFFFFF,
        _ptr(q, "q", _U8), _ptr(q_t, "q_t", _U8), _ptr(amax_out, "amax_out", torch.float32),
        _stream(stream)))
    return q, q_t, amax_out


def fp8_quantize_blocks(x: torch.Tensor, fmt: int, granularity: int, pow2: bool = False,
                        transpose: bool = False, stream=None):
    """Block cast; returns (q, scale_inv_blocks, q_t, scale_inv_blocks_t)."""
    rows, cols = x.shape
    q_t = torch.empty(cols, rows, dtype=torch.uint8, device=x.device) if transpose else None
    st = None
    if transpose:
        st = torch.empty(*_scale_shape_t(granularity, rows, cols), dtype=torch.float32,
                         device=x.device)
    q, q_t, s, _ = fp8_quantize(x, fmt, granularity, pow2=pow2, q_t=q_t, scale_inv_blocks_t=st,
                                stream=stream)
    return q, s, q_t, st


def _gemm_dims(A, B, layout):
    """(M, K, N) of A . B^T from the stored shapes: A [M,K] or, with
    LAYOUT_A_KM, [K,M]; B [N,K] or, with LAYOUT_B_KN, [K,N]."""
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = (A.shape[1], A.shape[0]) if int(layout) & LAYOUT_A_KM else A.shape
    N, Kb = (B.shape[1], B.shape[0]) if int(layout) & LAYOUT_B_KN else B.shape
    if Kb != K:
        raise ValueError("A and B disagree on K")
    return M, K, N


def fp8_gemm(A: torch.Tensor, fa: int, B: torch.Tensor, fb: int, scale_inv_a, scale_inv_b,
             ga: int = GRAN_TENSOR, gb: int = GRAN_TENSOR, out: int = OUT_BF16, D=None,
             accumulate: bool = False, layout: int = LAYOUT_TN, stream=None,
             bias=None) -> torch.Tensor:
    """D = (A . B^T) with dequantisation factors (+ bias [N], bf16); A [M,K],
    B [N,K] FP8 codes, or stored [K,M] / [K,N] per `layout`."""
    M, K, N = _gemm_dims(A, B, layout)
    if D is None:
        D = torch.empty(M, N, dtype=torch.bfloat16 if out == OUT_BF16 else torch.float32,
                        device=A.device)
    _check(lib().fp8_gemm(
        _ptr(A, "A", _U8), int(fa), _ptr(B, "B", _U8), int(fb), M, N, K, int(layout), int(ga),
        _ptr(scale_inv_a, "scale_inv_a", torch.float32), int(gb),
        _ptr(scale_inv_b, "scale_inv_b", torch.float32), _ptr(bias, "bias", torch.bfloat16),
        _ptr(D, "D", torch.bfloat16 if out == OUT_BF16 else torch.float32), int(out),
        int(bool(accumulate)), _stream(stream)))
    return D


def _gemm_args(A, fa, B, fb, scale_inv_a, scale_inv_b, ga=GRAN_TENSOR, gb=GRAN_TENSOR,
               out=OUT_BF16, D=None, accumulate=False, layout=LAYOUT_TN, bias=None):
    M, K, N = _gemm_dims(A, B, layout)
    if D is None:
        D = torch.empty(M, N, dtype=torch.bfloat16 if out == OUT_BF16 else torch.float32,
                        device=A.device)
    g = GemmArgsC(_ptr(A, "A", _U8), int(fa), _ptr(B, "B", _U8), int(fb), M, N, K, int(layout),
                  int(ga), _ptr(scale_inv_a, "scale_inv_a", torch.float32), int(gb),
                  _ptr(scale_inv_b, "scale_inv_b", torch.float32), _ptr(bias, "bias", torch.bfloat16),
                  _ptr(D, "D", torch.bfloat16 if out == OUT_BF16 else torch.float32), int(out),
                  int(bool(accumulate)))
    return g, D


def fp8_gemm_group(g1: dict, g2: dict, stream=None):
    """Two independent GEMMs in one launch; g1, g2 hold fp8_gemm's arguments
    by name (A, fa, B, fb, scale_inv_a, scale_inv_b and optionally ga, gb,
    out, D, accumulate, bias).  Returns (D1, D2)."""
    a1, D1 = _gemm_args(**g1)
    a2, D2 = _gemm_args(**g2)
    _check(lib().fp8_gemm_group(ctypes.byref(a1), ctypes.byref(a2), _stream(stream)))
    return D1, D2


def fp8_workspace_size(M: int, N: int, K: int, recipe: Recipe) -> int:
    return int(lib().fp8_workspace_size(M, N, K, ctypes.byref(recipe)))


def fp8_linear_fwd(X, W, recipe: Recipe, state: "LinearStateC", Y, workspace=None,
                   stream=None, bias=None) -> None:
    M, K = X.shape
    N = W.shape[0]
    _check(lib().fp8_linear_fwd(
        _ptr(X, "X", torch.bfloat16), _ptr(W, "W", torch.bfloat16),
        _ptr(bias, "bias", torch.bfloat16), M, N, K,
        ctypes.byref(recipe), ctypes.byref(state), _ptr(Y, "Y", torch.bfloat16),
        _ptr(workspace, "workspace"), 0 if workspace is None else workspace.numel(),
        _stream(stream)))


def fp8_linear_bwd(dY, M, N, K, recipe: Recipe, state: "LinearStateC", dX, dW,
                   accumulate_dW: bool, workspace, stream=None, dbias=None) -> None:
    _check(lib().fp8_linear_bwd(
        _ptr(dY, "dY", torch.bfloat16), M, N, K, ctypes.byref(recipe), ctypes.byref(state),
        _ptr(dX, "dX", torch.bfloat16), _ptr(dW, "dW", torch.float32), int(bool(accumulate_dW)),
        _ptr(dbias, "dbias", torch.float32),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))


def fp8_device_status(clear: bool = True) -> int:
    st = ctypes.c_int(0)
    _check(lib().fp8_device_status(ctypes.byref(st), int(bool(clear))))
    return st.value


STATUS_TIMEOUT = 1     # bit 0 of the device status word: a bounded wait gave up
STATUS_NONFINITE = 2   # bit 1: a scale update met a non-finite amax


def check_device_status() -> None:
    """Synchronise the device, read and clear the status word, and raise if a
    kernel reported a problem since the last read: Fp8Error with status
    FP8_ERR_TIMEOUT when a bounded wait gave up (that call's outputs are
    incomplete), else Fp8NumericsError when a scale update met a NaN or Inf
    (the previous scale was kept)."""
    st = fp8_device_status(clear=True)
    if st & STATUS_TIMEOUT:
        raise Fp8Error(-5, "a kernel's bounded wait gave up; its outputs are incomplete")
    if st & STATUS_NONFINITE:
        raise Fp8NumericsError("a scale update met a non-finite amax (NaN or Inf in a cast "
                               "tensor or its amax history); the previous scale was kept")


# ------------------------------------------------------------- layer object

class Fp8Linear:
    """One FP8 linear layer's device state (scales, histories, quantised
    operands, workspace), allocated with torch on `device`, plus fwd/bwd
    calls into the library.  `state_dict()` / `load_state_dict()` copy the
    scaling state for checkpoints.  With recipe.sr_grad the gradient cast
    rounds stochastically from the key (sr_seed, call counter).
    transposes (per-tensor recipes): keep transposed copies of the forward's
    codes for K-major backward GEMMs; by default (False) the backward reads
    the codes as stored (MN-major) and no copy is made.  The block-wise and
    per-row recipes always keep them (their transposed codes differ).
    check_status: after every forward / backward, synchronise and raise
    (check_device_status) if a kernel timed out or a scale update met a
    non-finite amax -- off by default, since it waits for the device."""

    def __init__(self, M: int, N: int, K: int, recipe: Recipe | None = None, device="cuda",
                 sr_seed: int = 0, transposes: bool = False, check_status: bool = False):
        self.M, self.N, self.K = M, N, K
        self.check_status = bool(check_status)
        self.recipe = recipe or Recipe()
        dev = torch.device(device)
        H = self.recipe.history_len if self.recipe.scaling == SCALING_DELAYED else 1
        f32 = dict(dtype=torch.float32, device=dev)
        self.scale = torch.ones(3, **f32)
        self.scale_inv = torch.ones(3, **f32)
        self.amax = torch.zeros(3, **f32)
        self.history = torch.zeros(3, H, **f32)
        self.pos = torch.zeros(3, dtype=torch.int32, device=dev)
        self.qscale_inv = torch.ones(2, **f32)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.x_q = torch.empty(M, K, **u8)
        self.w_q = torch.empty(N, K, **u8)
        block = self.recipe.scaling == SCALING_BLOCK
        rowwise = self.recipe.scaling == SCALING_ROW
        # block mode keeps the backward operands only when the token count
        # allows 1x128 blocks along it
        keep = (M % 128 == 0) if block else (rowwise or bool(transposes))
        self.x_qt = torch.empty(K, M, **u8) if keep else None
        self.w_qt = torch.empty(K, N, **u8) if keep else None
        self.x_sinv = self.w_sinv = self.x_sinv_t = self.w_sinv_t = None
        if block:
            self.x_sinv = torch.empty(M, K // 128, **f32)
            self.w_sinv = torch.empty(N // 128, K // 128, **f32)
            if keep:
                self.x_sinv_t = torch.empty(K, M // 128, **f32)
                self.w_sinv_t = torch.empty(K // 128, N // 128, **f32)
        elif rowwise:
            self.x_sinv = torch.empty(M, **f32)
            self.w_sinv = torch.empty(N, **f32)
            self.x_sinv_t = torch.empty(K, **f32)
            self.w_sinv_t = torch.empty(K, **f32)
        # (seed, counter) of the stochastic gradient cast, as two 64-bit words
        seed = int(sr_seed) & 0xFFFFFFFFFFFFFFFF
        self.sr_key = torch.tensor([seed - (1 << 64) if seed >> 63 else seed, 0],
                                   dtype=torch.int64, device=dev)
        ws = fp8_workspace_size(M, N, K, self.recipe)
        if self.recipe.scaling in (SCALING_DELAYED, SCALING_DYNAMIC) and not keep:
            ws -= (M * N + 255) // 256 * 256   # no dY_q^T: the backward reads dY_q MN-major
        self.workspace = torch.empty(max(ws, 16), **u8)
        p = lambda t: None if t is None else t.data_ptr()
        self.c_state = LinearStateC(p(self.scale), p(self.scale_inv), p(self.amax),
                                    p(self.history), p(self.pos), p(self.x_q), p(self.x_qt),
                                    p(self.w_q), p(self.w_qt), p(self.x_sinv), p(self.w_sinv),
                                    p(self.qscale_inv), p(self.x_sinv_t), p(self.w_sinv_t),
                                    p(self.sr_key))

    def forward(self, X: torch.Tensor, W: torch.Tensor, Y=None, stream=None,
                bias=None) -> torch.Tensor:
        """Y = X . W^T (+ bias [N], bf16)."""
        if Y is None:
            Y = torch.empty(self.M, self.N, dtype=torch.bfloat16, device=X.device)
        fp8_linear_fwd(X, W, self.recipe, self.c_state, Y, None, stream, bias=bias)
        if self.check_status:
            check_device_status()
        return Y

    def backward(self, dY: torch.Tensor, dX=None, dW=None, accumulate_dW: bool = False,
                 stream=None, dbias=None):
        """dX, dW (+)= ...; with dbias (fp32 [N]) also the bias gradient,
        accumulated like dW."""
        if dX is None:
            dX = torch.empty(self.M, self.K, dtype=torch.bfloat16, device=dY.device)
        if dW is None:
            dW = torch.zeros(self.N, self.K, dtype=torch.float32, device=dY.device)
        fp8_linear_bwd(dY, self.M, self.N, self.K, self.recipe, self.c_state, dX, dW,
                       accumulate_dW, self.workspace, stream, dbias=dbias)
        if self.check_status:
            check_device_status()
        return dX, dW

    def state_dict(self) -> dict:
        return {k: getattr(self, k).clone()
                for k in ("scale", "scale_inv", "amax", "history", "pos", "qscale_inv", "sr_key")}

    def load_state_dict(self, sd: dict) -> None:
        for k, v in sd.items():
            getattr(self, k).copy_(v)
