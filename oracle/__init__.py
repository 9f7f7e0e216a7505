"""CPU oracle for the scaled FP8 linear layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package.  The CUDA path never calls it and shares no code with it; the
two meet only through the seeded inputs of the ``synthetic`` package.

The arithmetic lives in ``fp8_oracle.c`` (plain C, fp64 GEMM accumulation,
bit-level FP8 codec); this module marshals numpy arrays into it and writes
the linear layer's forward/backward out as the pages' sequence of steps:

* "Mixed Precision LLM Training: The Complete Guide", section "Transformer
  Engine internals" > "Per-tensor scaling" / "Delayed scaling" /
  "History-based scaling" / "The HYBRID recipe" (E4M3 forward operands,
  E5M2 gradients, scale before the cast, inverse scales after the matmul,
  scale from the amax history applied one step late);
* same page, "DeepSeek FP8 training recipe" > "Block-wise scaling at 128
  granularity" (1x128 activation segments, 128x128 weight tiles, scales
  applied inside the matmul) and "Mixed-precision accumulation";
* same page, "FP8 and gradient accumulation" (FP32 wgrad buffer, upcast and
  add per micro-batch).

bf16 tensors cross this interface as ``numpy.uint16`` arrays of bit patterns.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

from . import build as _build

E4M3, E5M2 = 0, 1
ALGO_MAX, ALGO_MOST_RECENT = 0, 1
GRAN_TENSOR, GRAN_1x128, GRAN_128x128, GRAN_ROW = 0, 1, 2, 3
ROLE_X, ROLE_W, ROLE_DY = 0, 1, 2

_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is not None:
        return _lib
    L = ctypes.CDLL(_build.build())
    i64, c_int, c_float = ctypes.c_int64, ctypes.c_int, ctypes.c_float
    L.orc_decode.restype = ctypes.c_double
    L.orc_decode.argtypes = [ctypes.c_uint8, c_int]
    L.orc_encode.restype = ctypes.c_uint8
    L.orc_encode.argtypes = [c_float, c_int]
    L.orc_fp8_max.restype = ctypes.c_double
    L.orc_fp8_max.argtypes = [c_int]
    L.orc_decode_array.argtypes = [_u8p, i64, c_int, _f64p]
    L.orc_encode_array.argtypes = [_f32p, i64, c_int, _u8p]
    L.orc_amax_bf16.restype = c_float
    L.orc_amax_bf16.argtypes = [_u16p, i64]
    L.orc_update_scale.argtypes = [c_float, _f32p, _i32p, c_int, c_int, c_int, c_int, c_int,
                                   _f32p, _f32p]
    L.orc_quantize.argtypes = [_u16p, i64, i64, c_int, c_float, ctypes.c_void_p, ctypes.c_void_p]
    L.orc_block_quantize.argtypes = [_u16p, i64, i64, c_int, c_int, c_int, _u8p, _f32p]
    L.orc_row_quantize.argtypes = [_u16p, i64, i64, c_int, c_int, _u8p, _f32p]
    L.orc_gemm.argtypes = [_u8p, c_int, _u8p, c_int, i64, i64, i64, c_int, _f32p, c_int, _f32p,
                           _f64p, _f64p]
    L.orc_gemm_entries.argtypes = [_u8p, c_int, _u8p, c_int, i64, c_int, _f32p, c_int, _f32p,
                                   _i64p, _i64p, i64, _f64p, _f64p]
    L.orc_cast_counts.argtypes = [_u16p, i64, c_int, c_float,
                                  np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")]
    _u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
    L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
    L.orc_encode_sr.restype = ctypes.c_uint8
    L.orc_encode_sr.argtypes = [c_float, c_int, ctypes.c_uint32]
    L.orc_quantize_sr.argtypes = [_u16p, i64, i64, c_int, c_float, ctypes.c_uint64,
                                  ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
    L.orc_num_threads.restype = c_int
    _lib = L
    return L


def num_threads() -> int:
    return lib().orc_num_threads()


# ------------------------------------------------------------------ codec

def fp8_max(fmt: int) -> float:
    return lib().orc_fp8_max(fmt)


def decode(codes, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_decode_array(c.reshape(-1), c.size, fmt, out.reshape(-1))
    return out


def encode(values, fmt: int) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_encode_array(v.reshape(-1), v.size, fmt, out.reshape(-1))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- amax/scales

def amax(x_bits) -> np.float32:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    return np.float32(lib().orc_amax_bf16(x.reshape(-1), x.size))


@dataclass
class ScaleState:
    """Per-tensor scaling state of one tensor role: scale, its inverse, the
    amax history ring and its write position (initially 1, 1, zeros, 0)."""
    history_len: int
    scale: np.ndarray = field(default_factory=lambda: np.ones(1, np.float32))
    scale_inv: np.ndarray = field(default_factory=lambda: np.ones(1, np.float32))
    history: np.ndarray = None
    pos: np.ndarray = field(default_factory=lambda: np.zeros(1, np.int32))

    def __post_init__(self):
        if self.history is None:
            self.history = np.zeros(self.history_len, np.float32)

    def copy(self) -> "ScaleState":
        return ScaleState(self.history_len, self.scale.copy(), self.scale_inv.copy(),
                          self.history.copy(), self.pos.copy())


def update_scale(st: ScaleState, amax_value, algo: int, fmt: int, margin: int = 0,
                 pow2: bool = False) -> None:
    lib().orc_update_scale(float(amax_value), st.history, st.pos, st.history_len, algo, fmt,
                           int(margin), int(bool(pow2)), st.scale, st.scale_inv)


# ---------------------------------------------------------------- quantize

def quantize(x_bits, fmt: int, scale, transpose: bool = False):
    """Per-tensor quantisation of a 2-D bf16 tensor; returns (q, q_t or None)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    qt = np.empty((cols, rows), np.uint8) if transpose else None
    lib().orc_quantize(x, rows, cols, fmt, float(np.float32(scale)), q.ctypes.data,
                       qt.ctypes.data if transpose else None)
    return q, qt


def philox4x32_10(ctr, key):
    """Philox-4x32-10 of a 4-word counter and 2-word key -> 4 uint32 words."""
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def encode_sr(value, fmt: int, r32: int) -> int:
    return int(lib().orc_encode_sr(float(np.float32(value)), fmt, int(r32) & 0xFFFFFFFF))


def quantize_sr(x_bits, fmt: int, scale, seed: int, offset: int = 0, transpose: bool = False):
    """Per-tensor cast with stochastic rounding; returns (q, q_t or None)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    qt = np.empty((cols, rows), np.uint8) if transpose else None
    lib().orc_quantize_sr(x, rows, cols, fmt, float(np.float32(scale)), int(seed), int(offset),
                          q.ctypes.data, qt.ctypes.data if transpose else None)
    return q, qt


def row_quantize(x_bits, fmt: int, pow2: bool = False):
    """Per-row cast; returns (q, scale_inv[rows])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sinv = np.empty(rows, np.float32)
    lib().orc_row_quantize(x, rows, cols, fmt, int(bool(pow2)), q, sinv)
    return q, sinv


def cast_counts(x_bits, fmt: int, scale):
    """(underflow, saturated) counts of the per-tensor cast with `scale`."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    out = np.zeros(2, np.uint64)
    lib().orc_cast_counts(x, x.size, fmt, float(np.float32(scale)), out)
    return int(out[0]), int(out[1])


def block_quantize(x_bits, fmt: int, block_rows: int, pow2: bool = False):
    """Block quantisation (block_rows = 1 for 1x128, 128 for 128x128);
    returns (q, scale_inv[rows/block_rows, cols/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    assert cols % 128 == 0 and rows % block_rows == 0
    q = np.empty((rows, cols), np.uint8)
    sinv = np.empty((rows // block_rows, cols // 128), np.float32)
    lib().orc_block_quantize(x, rows, cols, fmt, block_rows, int(bool(pow2)), q, sinv)
    return q, sinv


# -------------------------------------------------------------------- GEMM

def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32).reshape(-1))


def _bias64(bias_bits):
    """A bf16 bias vector (bit patterns) as exact fp64 values."""
    return bf16_to_f32(np.ascontiguousarray(bias_bits, dtype=np.uint16)).astype(np.float64)


def gemm(A, fa: int, B, fb: int, sa, sb, ga: int = GRAN_TENSOR, gb: int = GRAN_TENSOR,
         bias=None):
    """D = A . B^T with dequantisation factors; A [M,K], B [N,K] FP8 codes.
    bias (bf16 bits [N], optional) is added to every row ("Transformer Engine
    internals": te.Linear's bias).  Returns (D, Dabs) in fp64, unrounded;
    Dabs is the sum of |products| that bounds the GEMM's rounding."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    D = np.empty((M, N), np.float64)
    Dabs = np.empty((M, N), np.float64)
    lib().orc_gemm(A, fa, B, fb, M, N, K, ga, _f32(sa), gb, _f32(sb), D, Dabs)
    if bias is not None:
        D = D + _bias64(bias)[None, :]
    return D, Dabs


def dbias(dY_bits):
    """Bias gradient: the column sums of dY [M x N] (the bias is added to
    every row, so its gradient sums the rows).  Returns (sum, sum of |.|) in
    fp64 over the exact bf16 values."""
    v = bf16_to_f32(np.ascontiguousarray(dY_bits, dtype=np.uint16)).astype(np.float64)
    return v.sum(axis=0), np.abs(v).sum(axis=0)


def gemm_entries(A, fa: int, B, fb: int, sa, sb, ii, jj, ga: int = GRAN_TENSOR,
                 gb: int = GRAN_TENSOR):
    """Entries D[ii[t], jj[t]] of A . B^T (for outputs too large to form)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    K = A.shape[1]
    assert B.shape[1] == K
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    D = np.empty(ii.shape[0], np.float64)
    Dabs = np.empty(ii.shape[0], np.float64)
    lib().orc_gemm_entries(A, fa, B, fb, K, ga, _f32(sa), gb, _f32(sb), ii, jj, ii.shape[0],
                           D, Dabs)
    return D, Dabs


# ------------------------------------------------------------------ linear

SCALING_DELAYED, SCALING_DYNAMIC, SCALING_BLOCK, SCALING_ROW = 0, 1, 2, 3


@dataclass
class Recipe:
    """HYBRID recipe: E4M3 forward operands, E5M2 gradients."""
    scaling: int = SCALING_DELAYED
    margin: int = 0
    history_len: int = 16
    algo: int = ALGO_MAX
    pow2: bool = False
    sr_grad: bool = False      # cast dY with stochastic rounding ("Stochastic rounding")


class LinearState:
    """The oracle's own scaling state for one linear layer (roles X, W, dY)
    plus the quantised forward operands that the backward pass reuses.  With
    recipe.sr_grad, backward call t casts dY with quantize_sr(seed=sr_seed,
    offset=t)."""

    def __init__(self, recipe: Recipe, sr_seed: int = 0):
        self.sr_seed = int(sr_seed)
        self.sr_counter = 0
        h = recipe.history_len if recipe.scaling == SCALING_DELAYED else 1
        self.roles = [ScaleState(h) for _ in range(3)]
        self.last_amax = np.zeros(3, np.float32)
        self.x_q = self.x_qt = self.w_q = self.w_qt = None
        self.x_sinv = self.w_sinv = None


def _per_tensor_operand(st: LinearState, role: int, x_bits, fmt: int, recipe: Recipe):
    rs = st.roles[role]
    a = amax(x_bits)
    st.last_amax[role] = a

    def cast(scale):
        if role == ROLE_DY and recipe.sr_grad:
            q, qt = quantize_sr(x_bits, fmt, scale, st.sr_seed, st.sr_counter, transpose=True)
            st.sr_counter += 1
            return q, qt
        return quantize(x_bits, fmt, scale, transpose=True)

    if recipe.scaling == SCALING_DYNAMIC:
        # current scaling: this tensor's own amax sets the scale it is cast with
        update_scale(rs, a, ALGO_MOST_RECENT, fmt, recipe.margin, recipe.pow2)
        q, qt = cast(rs.scale[0])
        return q, qt, rs.scale_inv.copy()
    # delayed: cast with the scale from earlier steps, then fold this amax in
    q, qt = cast(rs.scale[0])
    sinv = rs.scale_inv.copy()
    update_scale(rs, a, recipe.algo, fmt, recipe.margin, recipe.pow2)
    return q, qt, sinv


def linear_fwd(X_bits, W_bits, recipe: Recipe, st: LinearState, rows=None, bias=None):
    """Y = X . W^T (+ bias, bf16 bits [N]).  Returns (Y, Yabs) fp64 (all
    rows, or the listed rows)."""
    Y, Yabs = _linear_fwd(X_bits, W_bits, recipe, st, rows)
    if bias is not None:
        Y = Y + _bias64(bias)[None, :]
    return Y, Yabs


def _linear_fwd(X_bits, W_bits, recipe: Recipe, st: LinearState, rows):
    if recipe.scaling == SCALING_ROW:
        # per-token scales for X, per-output-channel scales for W; the
        # backward operands are the per-row casts of X^T and W^T (per-column
        # scales of X and W), since the row scales lie along the backward
        # reductions
        X = np.ascontiguousarray(X_bits, dtype=np.uint16)
        W = np.ascontiguousarray(W_bits, dtype=np.uint16)
        st.x_q, st.x_sinv = row_quantize(X, E4M3, recipe.pow2)
        st.w_q, st.w_sinv = row_quantize(W, E4M3, recipe.pow2)
        st.xt_q, st.xt_sinv = row_quantize(np.ascontiguousarray(X.T), E4M3, recipe.pow2)
        st.wt_q, st.wt_sinv = row_quantize(np.ascontiguousarray(W.T), E4M3, recipe.pow2)
        return _gemm_rows(st.x_q, E4M3, st.w_q, E4M3, st.x_sinv, st.w_sinv, rows, GRAN_ROW,
                          GRAN_ROW)
    if recipe.scaling == SCALING_BLOCK:
        X = np.ascontiguousarray(X_bits, dtype=np.uint16)
        st.x_q, st.x_sinv = block_quantize(X, E4M3, 1, recipe.pow2)
        st.w_q, st.w_sinv = block_quantize(W_bits, E4M3, 128, recipe.pow2)
        if X.shape[0] % 128 == 0:
            # backward operands: X^T cast in 1x128 blocks along the tokens, and
            # W_q^T, whose 128x128 blocks keep their scales
            st.xt_q, st.xt_sinv = block_quantize(np.ascontiguousarray(X.T), E4M3, 1, recipe.pow2)
            st.wt_q = np.ascontiguousarray(st.w_q.T)
            st.wt_sinv = np.ascontiguousarray(st.w_sinv.T)
        return _gemm_rows(st.x_q, E4M3, st.w_q, E4M3, st.x_sinv, st.w_sinv, rows,
                          GRAN_1x128, GRAN_128x128)
    st.x_q, st.x_qt, sx = _per_tensor_operand(st, ROLE_X, X_bits, E4M3, recipe)
    st.w_q, st.w_qt, sw = _per_tensor_operand(st, ROLE_W, W_bits, E4M3, recipe)
    st.sinv_fwd = (sx, sw)
    return _gemm_rows(st.x_q, E4M3, st.w_q, E4M3, sx, sw, rows)


def linear_bwd(dY_bits, recipe: Recipe, st: LinearState, dW_prev=None, rows_dx=None,
               rows_dw=None):
    """dX = dY . W  and  dW (+)= dY^T . X, E5M2 gradient, FP32 wgrad buffer.
    Returns ((dX, dXabs), (dW, dWabs)); dW includes dW_prev when given."""
    if recipe.scaling == SCALING_BLOCK:
        return _linear_bwd_block(dY_bits, recipe, st, dW_prev, rows_dx, rows_dw)
    if recipe.scaling == SCALING_ROW:
        dY = np.ascontiguousarray(dY_bits, dtype=np.uint16)
        dy_q, dy_s = row_quantize(dY, E5M2, recipe.pow2)
        dyt_q, dyt_s = row_quantize(np.ascontiguousarray(dY.T), E5M2, recipe.pow2)
        st.dy_q, st.dy_s, st.dyt_q, st.dyt_s = dy_q, dy_s, dyt_q, dyt_s
        dX = _gemm_rows(dy_q, E5M2, st.wt_q, E4M3, dy_s, st.wt_sinv, rows_dx, GRAN_ROW, GRAN_ROW)
        dW, dWabs = _gemm_rows(dyt_q, E5M2, st.xt_q, E4M3, dyt_s, st.xt_sinv, rows_dw, GRAN_ROW,
                               GRAN_ROW)
        if dW_prev is not None:
            prev = np.asarray(dW_prev, np.float64)
            dW = dW + (prev if rows_dw is None else prev[np.asarray(rows_dw)])
        return dX, (dW, dWabs)
    sx, sw = st.sinv_fwd
    dy_q, dy_qt, sdy = _per_tensor_operand(st, ROLE_DY, dY_bits, E5M2, recipe)
    st.dy_q, st.dy_qt, st.sinv_bwd = dy_q, dy_qt, sdy
    dX = _gemm_rows(dy_q, E5M2, st.w_qt, E4M3, sdy, sw, rows_dx)
    dW, dWabs = _gemm_rows(dy_qt, E5M2, st.x_qt, E4M3, sdy, sx, rows_dw)
    if dW_prev is not None:
        prev = np.asarray(dW_prev, np.float64)
        dW = dW + (prev if rows_dw is None else prev[np.asarray(rows_dw)])
    return dX, (dW, dWabs)


def _linear_bwd_block(dY_bits, recipe: Recipe, st: LinearState, dW_prev, rows_dx, rows_dw):
    """Block-wise backward ("DeepSeek FP8 training recipe" > "Block-wise
    scaling at 128 granularity"): dY in 1x128 blocks along N for dgrad (with
    W^T's 128x128 blocks), dY^T and X^T in 1x128 blocks along the tokens for
    wgrad; every 128-deep partial sum is scaled by its blocks' factors."""
    dY = np.ascontiguousarray(dY_bits, dtype=np.uint16)
    dy_q, dy_s = block_quantize(dY, E5M2, 1, recipe.pow2)
    dyt_q, dyt_s = block_quantize(np.ascontiguousarray(dY.T), E5M2, 1, recipe.pow2)
    st.dy_q, st.dy_s, st.dyt_q, st.dyt_s = dy_q, dy_s, dyt_q, dyt_s
    dX = _gemm_rows(dy_q, E5M2, st.wt_q, E4M3, dy_s, st.wt_sinv, rows_dx, GRAN_1x128,
                    GRAN_128x128)
    dW, dWabs = _gemm_rows(dyt_q, E5M2, st.xt_q, E4M3, dyt_s, st.xt_sinv, rows_dw, GRAN_1x128,
                           GRAN_1x128)
    if dW_prev is not None:
        prev = np.asarray(dW_prev, np.float64)
        dW = dW + (prev if rows_dw is None else prev[np.asarray(rows_dw)])
    return dX, (dW, dWabs)


def _gemm_rows(A, fa, B, fb, sa, sb, rows, ga=GRAN_TENSOR, gb=GRAN_TENSOR):
    if rows is None:
        return gemm(A, fa, B, fb, sa, sb, ga, gb)
    rows = np.asarray(rows, np.int64)
    N = B.shape[0]
    ii = np.repeat(rows, N)
    jj = np.tile(np.arange(N, dtype=np.int64), rows.shape[0])
    D, Dabs = gemm_entries(A, fa, B, fb, sa, sb, ii, jj, ga, gb)
    return D.reshape(rows.shape[0], N), Dabs.reshape(rows.shape[0], N)
