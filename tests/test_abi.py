"""The C-ABI library loads here (no GPU needed), exports every call that
include/fp8linear.h declares, and rejects invalid arguments on the host,
before any CUDA call, with the documented status codes."""
import ctypes
import os
import re

import pytest

import scaled_fp8_linear_gb300 as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(fp8_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_call():
    F.build()
    lib = F.lib()
    names = _declared()
    assert {"fp8_amax", "fp8_update_scale", "fp8_quantize", "fp8_gemm", "fp8_linear_fwd",
            "fp8_linear_bwd", "fp8_workspace_size", "fp8_last_error",
            "fp8_device_status"} <= names
    for n in names:
        assert hasattr(lib, n), n


def _header_constants():
    """Enumerators (NAME = value) and #defines of the public header."""
    src = open(os.path.join(ROOT, "include", "fp8linear.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    vals = {k: int(v) for k, v in re.findall(r"\b(FP8_[A-Z0-9_x]+)\s*=\s*(-?\d+)", src)}
    vals.update({k: int(v) for k, v in re.findall(r"#define\s+(FP8_[A-Z0-9_x]+)\s+(\d+)\b", src)})
    return vals


def test_binding_constants_match_the_header():
    """Every constant the binding exports under an FP8_ name of the header
    has the header's value (layouts, granularities, formats, recipes)."""
    hdr = _header_constants()
    checked = 0
    for name in F.__all__:
        if name.isupper() and "FP8_" + name in hdr:
            assert getattr(F, name) == hdr["FP8_" + name], name
            checked += 1
    for name in ("LAYOUT_TN", "LAYOUT_B_KN", "LAYOUT_A_KM", "LAYOUT_KM_KN", "GRAN_ROW",
                 "SCALE_POW2", "E4M3", "E5M2", "SCALING_DYNAMIC", "OUT_F32"):
        assert "FP8_" + name in hdr and getattr(F, name) == hdr["FP8_" + name], name
    assert checked >= 10


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced: every call below fails validation


def test_gemm_argument_checks():
    L = F.lib()
    one = ctypes.c_void_p(FAKE)
    ok = dict(A=one, fa=0, B=one, fb=0, M=128, N=128, K=128, layout=0, ga=0, sa=one, gb=0,
              sb=one, bias=None, D=one, out=0, acc=0, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return L.fp8_gemm(a["A"], a["fa"], a["B"], a["fb"], a["M"], a["N"], a["K"], a["layout"],
                          a["ga"], a["sa"], a["gb"], a["sb"], a["bias"], a["D"], a["out"], a["acc"],
                          a["s"])

    assert call(A=None) == -1
    assert call(fa=7) == -1
    assert call(layout=4) == -1 and call(layout=-1) == -1
    assert call(layout=F.LAYOUT_A_KM, M=200) == -2             # A stored [K x M]: M % 16 == 0
    assert call(layout=F.LAYOUT_B_KN, ga=F.GRAN_1x128, gb=F.GRAN_128x128) == -6   # block: TN only
    assert call(out=5) == -1
    assert call(acc=1) == -1                      # accumulate needs fp32 output
    assert call(N=120) == -2 and call(K=40) == -2  # not multiples of 16
    assert call(M=-1) == -2
    assert call(ga=1, K=144) == -2                 # block scales need K % 128 == 0
    # the power-of-two flag: only on block granularities; with it the block
    # shape rules still apply
    assert call(ga=F.GRAN_TENSOR | F.SCALE_POW2) == -1
    assert call(gb=F.GRAN_ROW | F.SCALE_POW2) == -1
    assert call(ga=F.GRAN_1x128 | F.SCALE_POW2, gb=F.GRAN_128x128 | F.SCALE_POW2, K=144) == -2
    assert call(ga=F.GRAN_128x128 | F.SCALE_POW2, gb=F.GRAN_128x128 | F.SCALE_POW2, M=200) == -2
    assert call(ga=F.GRAN_1x128 | F.SCALE_POW2, gb=F.GRAN_ROW) == -6   # block and per-row mixed
    assert call(ga=F.GRAN_1x128 | 32) == -1                             # unknown flag bits
    assert call(D=ctypes.c_void_p(FAKE + 4)) == -3
    assert "16-byte" in F.fp8_last_error()
    assert call(bias=ctypes.c_void_p(FAKE + 2)) == -3
    assert "bias" in F.fp8_last_error()


def test_quantize_update_amax_argument_checks():
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    # (x, rows, cols, fmt, gran, scale, pow2, q, q_t, sinv, sinv_t, amax, stream)
    assert L.fp8_quantize(None, 4, 4, 0, 0, p, 0, p, None, None, None, None, None) == -1
    assert L.fp8_quantize(p, 4, 4, 9, 0, p, 0, p, None, None, None, None, None) == -1
    assert L.fp8_quantize(p, 4, 4, 0, 0, None, 0, p, None, None, None, None, None) == -1  # no scale
    assert L.fp8_quantize(p, 24, 16, 0, 0, p, 0, p, p, None, None, None, None) == -2      # transpose rule
    assert L.fp8_quantize(p, 4, 100, 0, 1, None, 0, p, None, p, None, None, None) == -2   # cols % 128
    assert L.fp8_quantize(p, 100, 128, 0, 2, None, 0, p, None, p, None, None, None) == -2  # rows % 128
    assert L.fp8_quantize(p, 128, 128, 0, 1, p, 0, p, None, p, None, None, None) == -1    # scale in block mode
    assert L.fp8_quantize(p, 128, 128, 0, 1, None, 0, p, p, p, None, None, None) == -1    # q_t without sinv_t
    assert L.fp8_quantize(p, 100, 128, 0, 1, None, 0, p, p, p, p, None, None) == -2       # block q_t: rows % 128
    assert L.fp8_quantize(ctypes.c_void_p(FAKE + 2), 4, 4, 0, 0, p, 0, p, None, None, None, None, None) == -3
    assert L.fp8_update_scale(p, p, p, 0, 0, 0, 0, 0, p, p, None) == -1
    assert L.fp8_update_scale(p, p, p, 16, 0, 0, 65, 0, p, p, None) == -1
    assert L.fp8_update_scale(p, p, p, 16, 2, 0, 0, 0, p, p, None) == -1
    assert L.fp8_amax(p, -1, p, None) == -2
    assert L.fp8_amax(None, 4, p, None) == -1


def test_workspace_size_and_recipe_checks():
    r = F.Recipe()
    # codes of dY and dY^T, then the bias gradient's partial sums (N floats per 128 tokens)
    assert F.fp8_workspace_size(8192, 4096, 4096, r) == 2 * 8192 * 4096 + 64 * 4096 * 4
    assert F.fp8_workspace_size(16, 16, 16, r) == 2 * 256 + 256
    assert F.fp8_workspace_size(0, 16, 16, r) == 0
    # block: plus the 1x128 scale arrays of dY and dY^T
    assert F.fp8_workspace_size(256, 256, 256, F.Recipe(scaling=F.SCALING_BLOCK)) == \
        2 * 65536 + 2 * 2048 + 2 * 256 * 4
    assert F.fp8_workspace_size(16, 16, 16, F.Recipe(history_len=0)) == 0
    assert F.fp8_workspace_size(16, 16, 16, F.Recipe(margin=-1)) == 0
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    st = F.LinearStateC()
    bad = F.Recipe(history_len=2000)
    assert L.fp8_linear_fwd(p, p, None, 16, 16, 16, ctypes.byref(bad), ctypes.byref(st), p, None, 0, None) == -1
    blk = F.Recipe(scaling=F.SCALING_BLOCK)
    assert L.fp8_linear_fwd(p, p, None, 16, 16, 16, ctypes.byref(blk), ctypes.byref(st), p, None, 0, None) == -2
    # block-wise backward without the forward's transposed operands
    assert L.fp8_linear_bwd(p, 128, 128, 128, ctypes.byref(blk), ctypes.byref(st), p, p, 0, None, p, 1 << 20, None) == -1
    assert "x_qt" in F.fp8_last_error()
    r = F.Recipe()
    assert L.fp8_linear_fwd(p, p, None, 16, 16, 16, ctypes.byref(r), ctypes.byref(st), p, None, 0, None) == -1


def test_gemm_shapes_follow_the_layout():
    """The binding reads (M, K, N) from the stored shapes of each layout and
    refuses operands that disagree on K."""
    import torch
    a_mk = torch.zeros(48, 32, dtype=torch.uint8)      # [M x K]
    a_km = torch.zeros(32, 48, dtype=torch.uint8)      # [K x M]
    b_nk = torch.zeros(80, 32, dtype=torch.uint8)      # [N x K]
    b_kn = torch.zeros(32, 80, dtype=torch.uint8)      # [K x N]
    assert F._gemm_dims(a_mk, b_nk, F.LAYOUT_TN) == (48, 32, 80)
    assert F._gemm_dims(a_mk, b_kn, F.LAYOUT_B_KN) == (48, 32, 80)
    assert F._gemm_dims(a_km, b_nk, F.LAYOUT_A_KM) == (48, 32, 80)
    assert F._gemm_dims(a_km, b_kn, F.LAYOUT_KM_KN) == (48, 32, 80)
    for layout, a, b in ((F.LAYOUT_TN, a_mk, b_kn), (F.LAYOUT_B_KN, a_mk, b_nk),
                         (F.LAYOUT_A_KM, a_km, b_kn), (F.LAYOUT_KM_KN, a_mk, b_kn)):
        with pytest.raises(ValueError):
            F._gemm_dims(a, b, layout)


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        F.fp8_amax(x)


def test_quantize_counted_argument_checks():
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    # (x, rows, cols, fmt, scale, q, q_t, amax, counts, stream)
    assert L.fp8_quantize_counted(p, 4, 4, 0, p, p, None, None, None, None) == -1     # no counts
    assert L.fp8_quantize_counted(p, 4, 4, 0, None, p, None, None, p, None) == -1     # no scale
    assert L.fp8_quantize_counted(p, 4, 4, 0, p, p, None, None, ctypes.c_void_p(FAKE + 4), None) == -3


def test_quantize_sr_argument_checks():
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    # (x, rows, cols, fmt, scale, seed, offset, q, q_t, amax, stream)
    assert L.fp8_quantize_sr(p, 4, 4, 0, None, 1, 0, p, None, None, None) == -1       # no scale
    assert L.fp8_quantize_sr(p, 4, 4, 2, p, 1, 0, p, None, None, None) == -1          # format
    assert L.fp8_quantize_sr(None, 4, 4, 0, p, 1, 0, p, None, None, None) == -1      # no x
    assert L.fp8_quantize_sr(p, -1, 4, 0, p, 1, 0, p, None, None, None) == -2         # shape
    assert L.fp8_quantize_sr(p, 4, 24, 0, p, 1, 0, p, p, None, None) == -2            # q_t needs %16
    assert L.fp8_quantize_sr(ctypes.c_void_p(FAKE + 2), 4, 4, 0, p, 1, 0, p, None, None, None) == -3
    assert "fp8_quantize" in F.fp8_last_error()


def test_bias_argument_checks():
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    r = F.Recipe()
    # a state whose every pointer is set (never dereferenced: the calls fail validation)
    st = F.LinearStateC(*([FAKE] * len(F.LinearStateC._fields_)))
    odd = ctypes.c_void_p(FAKE + 2)
    assert L.fp8_linear_fwd(p, p, odd, 16, 16, 16, ctypes.byref(r), ctypes.byref(st), p, None, 0, None) == -3
    ws = F.fp8_workspace_size(256, 256, 256, r)
    ws_operands = 2 * 256 * 256
    # dbias needs the partial-sum part of the workspace; without dbias the operands suffice
    assert L.fp8_linear_bwd(p, 256, 256, 256, ctypes.byref(r), ctypes.byref(st), p, p, 0, p, p,
                            ws_operands, None) == -1
    assert "workspace" in F.fp8_last_error()
    assert L.fp8_linear_bwd(p, 256, 256, 256, ctypes.byref(r), ctypes.byref(st), p, p, 0,
                            ctypes.c_void_p(FAKE + 1), p, ws, None) == -3


def test_sr_grad_recipe_checks():
    L = F.lib()
    p = ctypes.c_void_p(FAKE)
    st = F.LinearStateC(*([FAKE] * (len(F.LinearStateC._fields_) - 1) + [None]))
    assert F.fp8_workspace_size(256, 256, 256, F.Recipe(sr_grad=True)) > 0
    # stochastic dY rounding is built for per-tensor scaling only
    for mode in (F.SCALING_BLOCK, F.SCALING_ROW):
        r = F.Recipe(scaling=mode, sr_grad=True)
        assert F.fp8_workspace_size(256, 256, 256, r) == 0
        assert L.fp8_linear_fwd(p, p, None, 256, 256, 256, ctypes.byref(r), ctypes.byref(st),
                                p, None, 0, None) == -6
    bad = F.Recipe(sr_grad=True)
    bad.sr_grad = 2
    assert L.fp8_linear_fwd(p, p, None, 256, 256, 256, ctypes.byref(bad), ctypes.byref(st),
                            p, None, 0, None) == -1
    # the backward needs the state's key
    r = F.Recipe(sr_grad=True)
    ws = F.fp8_workspace_size(256, 256, 256, r)
    assert L.fp8_linear_bwd(p, 256, 256, 256, ctypes.byref(r), ctypes.byref(st), p, p, 0, None,
                            p, ws, None) == -1
    assert "sr_key" in F.fp8_last_error()


def test_gemm_group_argument_checks():
    L = F.lib()
    one = ctypes.c_void_p(FAKE)
    good = F.GemmArgsC(one, 0, one, 0, 256, 256, 256, 0, 0, one, 0, one, None, one, 0, 0)
    bad = F.GemmArgsC(one, 0, one, 0, 256, 120, 256, 0, 0, one, 0, one, None, one, 0, 0)
    assert L.fp8_gemm_group(None, ctypes.byref(good), None) == -1
    assert L.fp8_gemm_group(ctypes.byref(good), None, None) == -1
    assert L.fp8_gemm_group(ctypes.byref(good), ctypes.byref(bad), None) == -2   # N % 16
    odd_bias = F.GemmArgsC(one, 0, one, 0, 256, 256, 256, 0, 0, one, 0, one,
                           ctypes.c_void_p(FAKE + 2), one, 0, 0)
    assert L.fp8_gemm_group(ctypes.byref(odd_bias), ctypes.byref(good), None) == -3


def test_noalloc_checks_arguments_before_touching_the_device():
    """fp8_linear_bwd_noalloc validates everything before it looks up its
    scratch array: on a machine without a GPU an invalid call still returns
    its own status, not a CUDA error from the lookup."""
    L = F.lib()
    fn = L.fp8_linear_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                   ctypes.POINTER(F.Recipe), ctypes.POINTER(F.LinearStateC), ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    p = ctypes.c_void_p(FAKE)
    st = F.LinearStateC(*([FAKE] * len(F.LinearStateC._fields_)))
    bad = F.Recipe(history_len=0)
    assert fn(p, 256, 256, 256, ctypes.byref(bad), ctypes.byref(st), p, p, 0, None) == -1
    assert fn(p, 256, 120, 256, ctypes.byref(F.Recipe()), ctypes.byref(st), p, p, 0, None) == -2
    assert fn(p, 256, 256, 256, ctypes.byref(F.Recipe()), ctypes.byref(st),
              ctypes.c_void_p(FAKE + 2), p, 0, None) == -3
    blk = F.Recipe(scaling=F.SCALING_BLOCK)
    assert fn(p, 256, 256, 256, ctypes.byref(blk), ctypes.byref(F.LinearStateC()), p, p, 0,
              None) == -1
    # a shape whose dY operands exceed the scratch: -2 with the limit named
    assert fn(p, 8192, 8192, 4096, ctypes.byref(F.Recipe()), ctypes.byref(st), p, p, 0,
              None) == -2
    assert "scratch" in F.fp8_last_error()


def test_epilogue_wait_hook_refuses_a_longer_limit():
    fn = F.lib().fp8_test_set_epilogue_wait_ns
    fn.argtypes = [ctypes.c_uint64]
    fn.restype = ctypes.c_int
    assert fn(2_000_000_001) == -1
    assert "2 s" in F.fp8_last_error()
