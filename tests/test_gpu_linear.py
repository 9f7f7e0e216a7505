"""GPU parity of the composed linear layer (fp8_linear_fwd / fp8_linear_bwd)
against the oracle's own state machine: quantised operands, amaxes, scales
and histories bit-exact at every step; Y, dX, dW within the GEMM bound.
The last tests run the full-size workload shapes and check sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import scaled_fp8_linear_gb300 as F
import synthetic
from tests.helpers import assert_gemm_bound, bits, f32bits, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    F.build()
    F.lib()
    yield
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0


def _orecipe(r: F.Recipe) -> oracle.Recipe:
    return oracle.Recipe(scaling=r.scaling, margin=r.margin, history_len=r.history_len,
                         algo=r.amax_algo, pow2=bool(r.pow2))


def _check_state(layer, ost, roles=(0, 1, 2)):
    for r in roles:
        rs = ost.roles[r]
        assert f32bits(layer.scale[r].cpu().numpy()) == f32bits(rs.scale[0]), r
        assert f32bits(layer.scale_inv[r].cpu().numpy()) == f32bits(rs.scale_inv[0]), r
        assert np.array_equal(f32bits(layer.history[r].cpu().numpy()), f32bits(rs.history)), r
        assert layer.pos[r].item() == rs.pos[0]


@pytest.mark.parametrize("recipe", [
    F.Recipe(F.SCALING_DELAYED, history_len=16),
    F.Recipe(F.SCALING_DELAYED, history_len=4, amax_algo=F.AMAX_MOST_RECENT, margin=1),
    F.Recipe(F.SCALING_DELAYED, history_len=16, pow2=True),
    F.Recipe(F.SCALING_DYNAMIC)], ids=["delayed16", "delayed4_recent_m1", "delayed16_pow2", "dynamic"])
@pytest.mark.parametrize("transposes", [False, True], ids=["mn_major", "transposed_copies"])
def test_training_steps(recipe, transposes):
    """20 steps (wrapping a 16-long history), fresh seeded X, dY each step,
    fixed W; wgrad accumulated over pairs of steps (two micro-batches).  The
    backward reads the forward's codes as stored, or transposed copies."""
    M, N, K = 256, 384, 512
    layer = F.Fp8Linear(M, N, K, recipe, device=DEV, transposes=transposes)
    orec = _orecipe(recipe)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=1000)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    dW_o = np.zeros((N, K))
    for step in range(20):
        X = synthetic.with_outlier_channels((M, K), 1.0, 4, 50.0 if step % 5 else 200.0, seed=step)
        dY = synthetic.normal((M, N), 1e-3 * (1 + step % 3), seed=100 + step)
        if step == 7:
            dY.zero_()                        # all-zero gradient: its scale update is skipped
        acc = step % 2 == 1
        Y = layer.forward(X.to(DEV), W.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW, accumulate_dW=acc)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost)
        prev = dW_o.copy()
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost,
                                                       dW_prev=prev if acc else None)
        assert np.array_equal(u8(layer.x_q), ost.x_q), step
        assert np.array_equal(u8(layer.w_q), ost.w_q), step
        if transposes:
            assert np.array_equal(u8(layer.w_qt), ost.w_qt), step
            assert np.array_equal(u8(layer.x_qt), ost.x_qt), step
        else:
            assert layer.x_qt is None and layer.w_qt is None
        assert np.array_equal(f32bits(layer.amax.cpu().numpy()), f32bits(ost.last_amax)), step
        assert np.array_equal(f32bits(layer.qscale_inv.cpu().numpy()),
                              f32bits(np.concatenate(ost.sinv_fwd))), step
        _check_state(layer, ost)
        assert_gemm_bound(Y, Yo, Yabs, what=f"Y step {step}")
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, prev=prev if acc else None, what=f"dW step {step}")
        dW_o = dW.cpu().numpy().astype(np.float64)   # next step accumulates onto the GPU buffer


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (1024, 1040, 1024), (1008, 1024, 1040),
                                   (32, 64, 48)],
                         ids=["all_at_limit", "w_and_dy_over", "x_under_w_over", "tiny"])
def test_dynamic_small_tensor_path(M, N, K):
    """Dynamic scaling of tensors of at most 2^20 elements takes the one-launch
    small-tensor cast (one cluster per tensor); larger ones the amax pass and
    the chunked cast.  Either way, at and across the limit: the codes of X, W
    and dY, every amax, scale and history bit-exact; Y, dX, dW within the
    bound; 3 steps, the last with an all-zero dY (its scale update skipped)."""
    rec = F.Recipe(F.SCALING_DYNAMIC)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=51)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    for step in range(3):
        X = synthetic.with_outlier_channels((M, K), 1.0, 3, 40.0, seed=60 + step)
        dY = synthetic.normal((M, N), 1e-3, seed=70 + step)
        if step == 2:
            dY.zero_()
        Y = layer.forward(X.to(DEV), W.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost)
        assert np.array_equal(u8(layer.x_q), ost.x_q), step
        assert np.array_equal(u8(layer.w_q), ost.w_q), step
        assert np.array_equal(u8(layer.workspace[:M * N]).reshape(M, N), ost.dy_q), step
        assert np.array_equal(f32bits(layer.amax.cpu().numpy()), f32bits(ost.last_amax)), step
        _check_state(layer, ost)
        assert_gemm_bound(Y, Yo, Yabs, what=f"Y step {step}")
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, what=f"dW step {step}")


@pytest.mark.parametrize("M,N,K,with_bias,fmt", [
    (256, 512, 512, False, F.E4M3), (128, 128, 128, True, F.E4M3), (1024, 128, 768, False, F.E4M3),
    (112, 1024, 64, True, F.E4M3), (208, 400, 336, True, F.E5M2), (16, 16, 16, False, F.E5M2)],
    ids=["small_case_2x4_tiles", "one_tile_bias", "8x1_tiles_k768", "1x8_tiles_ragged_m_bias",
         "ragged_k336_bias_e5m2", "smallest_e5m2"])
def test_dynamic_small_forward_shapes(M, N, K, with_bias, fmt):
    """Small dynamic forwards (the one-launch small-tensor cast, then the
    GEMM) over 1 to 8 output tiles, ragged M, N and K, with and without bias,
    E4M3 and E5M2 forward operands.  Over 3 steps, the last with an all-zero
    X (its scale update skipped): the codes of X and W (which the backward
    reads), every amax, scale and history bit-exact against the oracle; Y
    within the bound.  With E4M3 forward operands the backward after each
    forward stays in parity too."""
    rec = F.Recipe(F.SCALING_DYNAMIC, fwd_format=fmt)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    W = synthetic.normal((N, K), 0.02, seed=81)
    b = synthetic.normal((N,), 0.1, seed=82) if with_bias else None
    hybrid = fmt == F.E4M3
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    rx, rw = oracle.ScaleState(1), oracle.ScaleState(1)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    for step in range(3):
        X = synthetic.with_outlier_entries((M, K), 1.0, 0.001, 50.0, seed=90 + step)
        if step == 2:
            X.zero_()
        Y = layer.forward(X.to(DEV), W.to(DEV), bias=b.to(DEV) if with_bias else None)
        ax, aw = oracle.amax(bits(X)), oracle.amax(bits(W))
        if hybrid:
            Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost,
                                         bias=bits(b) if with_bias else None)
            xq, wq = ost.x_q, ost.w_q
            _check_state(layer, ost, roles=(0, 1))
        else:
            oracle.update_scale(rx, ax, oracle.ALGO_MOST_RECENT, fmt)
            oracle.update_scale(rw, aw, oracle.ALGO_MOST_RECENT, fmt)
            xq, _ = oracle.quantize(bits(X), fmt, rx.scale[0])
            wq, _ = oracle.quantize(bits(W), fmt, rw.scale[0])
            Yo, Yabs = oracle.gemm(xq, fmt, wq, fmt, rx.scale_inv, rw.scale_inv,
                                   bias=bits(b) if with_bias else None)
            for r, rs in ((0, rx), (1, rw)):
                assert f32bits(layer.scale[r].cpu().numpy()) == f32bits(rs.scale[0]), (step, r)
                assert f32bits(layer.scale_inv[r].cpu().numpy()) == f32bits(rs.scale_inv[0]), (step, r)
                assert np.array_equal(f32bits(layer.history[r].cpu().numpy()), f32bits(rs.history))
        assert np.array_equal(u8(layer.x_q), xq), step
        assert np.array_equal(u8(layer.w_q), wq), step
        am = layer.amax.cpu().numpy()
        assert f32bits(am[0]) == f32bits(np.float32(ax)) and f32bits(am[1]) == f32bits(np.float32(aw))
        assert_gemm_bound(Y, Yo, Yabs, what=f"Y step {step}")
        if hybrid:
            dY = synthetic.normal((M, N), 1e-3, seed=95 + step)
            dX, _ = layer.backward(dY.to(DEV), dW=dW)
            (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost)
            assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
            assert_gemm_bound(dW, dWo, dWabs, what=f"dW step {step}")


@pytest.mark.parametrize("recipe,transposes", [
    (F.Recipe(F.SCALING_DYNAMIC), False), (F.Recipe(F.SCALING_DYNAMIC), True),
    (F.Recipe(F.SCALING_DELAYED, history_len=4), False),
    (F.Recipe(F.SCALING_DYNAMIC, sr_grad=True), False),
    (F.Recipe(F.SCALING_BLOCK), False), (F.Recipe(F.SCALING_ROW), False)],
    ids=["dynamic", "dynamic_transposed_copies", "delayed4", "dynamic_sr_grad", "block", "row"])
def test_empty_token_batch(recipe, transposes):
    """A batch without tokens (M = 0: an expert that received none): X, Y, dY
    and dX are empty (NULL pointers), the forward still casts W, the scaling
    state advances as the oracle's does (X's and dY's amax are 0, so their
    scale updates are skipped), dW and dbias come out zero, and with
    accumulation stay as they were; over 2 steps, no device error."""
    M, N, K = 0, 384, 256
    layer = F.Fp8Linear(M, N, K, recipe, device=DEV, transposes=transposes)
    orec = oracle.Recipe(scaling=recipe.scaling, margin=recipe.margin,
                         history_len=recipe.history_len, algo=recipe.amax_algo,
                         pow2=bool(recipe.pow2), sr_grad=bool(recipe.sr_grad))
    ost = oracle.LinearState(orec)
    per_tensor = recipe.scaling in (F.SCALING_DELAYED, F.SCALING_DYNAMIC)
    W = synthetic.normal((N, K), 0.02, seed=5)
    X = torch.empty(M, K, dtype=torch.bfloat16)
    dY = torch.empty(M, N, dtype=torch.bfloat16)
    dW = torch.full((N, K), 3.0, dtype=torch.float32, device=DEV)
    db = torch.full((N,), 2.0, dtype=torch.float32, device=DEV)
    for step in range(2):
        acc = step > 0
        prev_w, prev_b = dW.clone(), db.clone()
        Y = layer.forward(X.to(DEV), W.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW, dbias=db, accumulate_dW=acc)
        torch.cuda.synchronize()
        assert Y.shape == (0, N) and dX.shape == (0, K)
        oracle.linear_fwd(bits(X), bits(W), orec, ost)
        oracle.linear_bwd(bits(dY), orec, ost)
        assert np.array_equal(u8(layer.w_q), ost.w_q), step
        if per_tensor:
            _check_state(layer, ost)
            assert np.array_equal(f32bits(layer.amax.cpu().numpy()), f32bits(ost.last_amax)), step
        else:
            assert np.array_equal(f32bits(layer.w_sinv.cpu().numpy().reshape(-1)),
                                  f32bits(np.asarray(ost.w_sinv).reshape(-1))), step
        if acc:
            assert torch.equal(dW, prev_w) and torch.equal(db, prev_b), step
        else:
            assert not torch.any(dW) and not torch.any(db), step


@pytest.mark.parametrize("M,N,K,with_bias,transposes", [
    (656, 272, 400, False, False), (656, 272, 400, True, False), (272, 656, 400, False, False),
    (656, 272, 400, True, True), (48, 272, 400, True, False), (656, 48, 400, False, False)],
    ids=["x_larger", "x_larger_dbias", "w_larger", "x_larger_dbias_transposes", "few_tokens_dbias",
         "few_features"])
def test_dynamic_ragged(M, N, K, with_bias, transposes):
    """Dynamic scaling with X or W the larger operand and ragged tiles in
    every dimension (fewer than 256 tokens or output features included):
    codes (and transposed copies), amaxes and scales bit-exact, Y / dX / dW
    (and dbias) within the bound, over 2 steps."""
    rec = F.Recipe(F.SCALING_DYNAMIC)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV, transposes=transposes)
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=21)
    b = synthetic.normal((N,), 0.1, seed=22) if with_bias else None
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    for step in range(2):
        X = synthetic.with_outlier_channels((M, K), 1.0, 3, 40.0, seed=30 + step)
        dY = synthetic.normal((M, N), 1e-3, seed=40 + step)
        db = torch.zeros(N, dtype=torch.float32, device=DEV) if with_bias else None
        Y = layer.forward(X.to(DEV), W.to(DEV), bias=b.to(DEV) if with_bias else None)
        dX, _ = layer.backward(dY.to(DEV), dW=dW, dbias=db)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost,
                                     bias=bits(b) if with_bias else None)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost)
        pairs = [(layer.x_q, ost.x_q), (layer.w_q, ost.w_q)]
        if transposes:
            pairs += [(layer.x_qt, ost.x_qt), (layer.w_qt, ost.w_qt)]
        for got, want in pairs:
            assert np.array_equal(u8(got), want), step
        assert np.array_equal(f32bits(layer.amax.cpu().numpy()), f32bits(ost.last_amax)), step
        _check_state(layer, ost)
        assert_gemm_bound(Y, Yo, Yabs, what=f"Y step {step}")
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, what=f"dW step {step}")
        if with_bias:   # fp32 column sums of 128-row partials, in order
            want, wabs = oracle.dbias(bits(dY))
            err = np.abs(db.cpu().numpy().astype(np.float64) - want)
            assert np.all(err <= (16 + (M + 127) // 128) * 2.0 ** -24 * wabs), step


def test_block_forward():
    M, N, K = 300, 512, 768
    rec = F.Recipe(F.SCALING_BLOCK)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    X = synthetic.student_t_rows((M, K), 1.0, 3, seed=5)
    W = synthetic.student_t_rows((N, K), 0.02, 3, seed=6)
    Y = layer.forward(X.to(DEV), W.to(DEV))
    ost = oracle.LinearState(_orecipe(rec))
    Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), _orecipe(rec), ost)
    assert np.array_equal(u8(layer.x_q), ost.x_q)
    assert np.array_equal(u8(layer.w_q), ost.w_q)
    assert np.array_equal(f32bits(layer.x_sinv.cpu().numpy()), f32bits(ost.x_sinv))
    assert np.array_equal(f32bits(layer.w_sinv.cpu().numpy()), f32bits(ost.w_sinv))
    assert_gemm_bound(Y, Yo, Yabs)


def _align256(n):
    return (n + 255) // 256 * 256


def _check_block_dy(layer, ost, M, N):
    """The block-wise backward's dY casts, as the workspace holds them: dY_q
    [M x N] with its 1x128 scales [M][N/128] along N, and dY_q^T [N x M] with
    its 1x128 scales [N][M/128] along the tokens -- bit-exact against the
    oracle's block casts of dY and dY^T."""
    ws = layer.workspace
    mn = M * N
    o_qt, o_s = _align256(mn), 2 * _align256(mn)
    o_st = o_s + _align256(4 * (mn // 128))
    assert np.array_equal(u8(ws[:mn]).reshape(M, N), ost.dy_q)
    assert np.array_equal(u8(ws[o_qt:o_qt + mn]).reshape(N, M), ost.dyt_q)
    s = ws[o_s:o_s + 4 * (mn // 128)].view(torch.float32).cpu().numpy().reshape(M, N // 128)
    st = ws[o_st:o_st + 4 * (mn // 128)].view(torch.float32).cpu().numpy().reshape(N, M // 128)
    assert np.array_equal(f32bits(s), f32bits(ost.dy_s))
    assert np.array_equal(f32bits(st), f32bits(ost.dyt_s))


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (1024, 768, 1280), (640, 896, 384)])
@pytest.mark.parametrize("pow2", [False, True], ids=["fp32_scales", "pow2_scales"])
def test_block_training_steps(M, N, K, pow2):
    """Block-wise forward + backward over 3 steps, wgrad accumulated: every
    quantised operand and block scale bit-exact, Y / dX / dW within the
    bound.  With pow2 the three GEMMs run on the block-scaled MMA."""
    rec = F.Recipe(F.SCALING_BLOCK, pow2=pow2)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    W = synthetic.student_t_rows((N, K), 0.02, 3, seed=77)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    dW_o = np.zeros((N, K))
    for step in range(3):
        X = synthetic.student_t_rows((M, K), 1.0, 3, seed=step)
        dY = synthetic.normal((M, N), 1e-3 * (1 + step), seed=40 + step)
        acc = step > 0
        Y = layer.forward(X.to(DEV), W.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW, accumulate_dW=acc)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost)
        prev = dW_o.copy()
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost,
                                                       dW_prev=prev if acc else None)
        assert np.array_equal(u8(layer.x_q), ost.x_q)
        assert np.array_equal(u8(layer.x_qt), ost.xt_q)
        assert np.array_equal(f32bits(layer.x_sinv_t.cpu().numpy()), f32bits(ost.xt_sinv))
        assert np.array_equal(u8(layer.w_qt), ost.wt_q)
        assert np.array_equal(f32bits(layer.w_sinv_t.cpu().numpy()), f32bits(ost.wt_sinv))
        _check_block_dy(layer, ost, M, N)
        assert_gemm_bound(Y, Yo, Yabs, what=f"Y step {step}")
        assert_gemm_bound(dX, dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(dW, dWo, dWabs, prev=prev if acc else None, what=f"dW step {step}")
        dW_o = dW.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (4096, 2048, 1024)])
def test_row_training_steps(M, N, K):
    """Per-row (per-token / per-channel) scaling, forward + backward, 2 steps
    with wgrad accumulation: casts and scales bit-exact, GEMMs within the
    bound."""
    rec = F.Recipe(F.SCALING_ROW)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    W = synthetic.student_t_rows((N, K), 0.02, 3, seed=91)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    dW_o = np.zeros((N, K))
    rows = None if M * N <= 256 * 384 else np.arange(0, M, 97)
    for step in range(2):
        X = synthetic.with_outlier_channels((M, K), 1.0, 4, 50.0, seed=60 + step)
        dY = synthetic.normal((M, N), 1e-3, seed=70 + step)
        acc = step > 0
        Y = layer.forward(X.to(DEV), W.to(DEV))
        dX, _ = layer.backward(dY.to(DEV), dW=dW, accumulate_dW=acc)
        Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost, rows=rows)
        prev = dW_o.copy()
        rows_dw = None if rows is None else np.arange(0, N, 53)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(
            bits(dY), orec, ost, dW_prev=prev if acc else None, rows_dx=rows, rows_dw=rows_dw)
        for got, want in ((layer.x_q, ost.x_q), (layer.w_q, ost.w_q), (layer.x_qt, ost.xt_q),
                          (layer.w_qt, ost.wt_q)):
            assert np.array_equal(u8(got), want)
        for got, want in ((layer.x_sinv, ost.x_sinv), (layer.w_sinv, ost.w_sinv),
                          (layer.x_sinv_t, ost.xt_sinv), (layer.w_sinv_t, ost.wt_sinv)):
            assert np.array_equal(f32bits(got.cpu().numpy()), f32bits(want))
        sel = (lambda t, r: t if r is None else t[torch.as_tensor(r, device=DEV)])
        assert_gemm_bound(sel(Y, rows), Yo, Yabs, what=f"Y step {step}")
        assert_gemm_bound(sel(dX, rows), dXo, dXabs, what=f"dX step {step}")
        assert_gemm_bound(sel(dW, rows_dw), dWo, dWabs,
                          prev=(prev if rows_dw is None else prev[rows_dw]) if acc else None,
                          what=f"dW step {step}")
        dW_o = dW.cpu().numpy().astype(np.float64)


def test_checkpoint_restore_gives_identical_next_step():
    M, N, K = 128, 256, 256
    rec = F.Recipe(F.SCALING_DELAYED, history_len=16)
    a = F.Fp8Linear(M, N, K, rec, device=DEV)
    W = synthetic.normal((N, K), 0.02, seed=1).to(DEV)
    for s in range(5):
        a.forward(synthetic.normal((M, K), 1.0 + s, seed=s).to(DEV), W)
        a.backward(synthetic.normal((M, N), 1e-3, seed=50 + s).to(DEV))
    sd = a.state_dict()
    b = F.Fp8Linear(M, N, K, rec, device=DEV)
    b.load_state_dict(sd)
    X = synthetic.normal((M, K), 9.0, seed=99).to(DEV)
    ya, yb = a.forward(X, W), b.forward(X, W)
    assert torch.equal(ya, yb)
    assert torch.equal(a.scale, b.scale) and torch.equal(a.history, b.history)


# ----------------------------------------------------------- full-size shapes

LINEARS_7B = [("qkv", 4096, 12288), ("o", 4096, 4096), ("gate", 4096, 11008),
              ("up", 4096, 11008), ("down", 11008, 4096)]
LINEARS_70B = [("qkv", 8192, 10240), ("o", 8192, 8192), ("gate", 8192, 28672),
               ("up", 8192, 28672), ("down", 28672, 8192)]
SAMPLE = 64   # seeded rows and full columns checked per GEMM output


def _sample(n, k, seed):
    """k distinct sorted indices of 0..n-1 (the first and last included)."""
    rng = np.random.default_rng(seed)
    inner = rng.choice(np.arange(1, n - 1), min(k, n) - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], inner])).astype(np.int64)


def _columns(A, fa, B, fb, sa, sb, nrows, cols, ga=oracle.GRAN_TENSOR, gb=oracle.GRAN_TENSOR):
    """Full columns `cols` of A . B^T (all nrows rows) from the oracle's
    codes and factors, as [nrows x len(cols)]."""
    ii = np.repeat(np.arange(nrows, dtype=np.int64), len(cols))
    jj = np.tile(cols, nrows)
    D, Dabs = oracle.gemm_entries(A, fa, B, fb, sa, sb, ii, jj, ga, gb)
    return D.reshape(nrows, len(cols)), Dabs.reshape(nrows, len(cols))


def _outlier_channels(K):
    return 43 if K == 11008 else max(1, K // 256)


FULL_CASES = (
    [(f"llama2-7b {n}, delayed", 8192, N, K, F.SCALING_DELAYED, False, 1)
     for n, K, N in LINEARS_7B]
    + [("llama2-7b qkv, delayed, transposed copies", 8192, 12288, 4096, F.SCALING_DELAYED,
        True, 1)]
    + [(f"llama2-70b {n}, dynamic, 2 micro-batches", 4096, N, K, F.SCALING_DYNAMIC, False, 2)
       for n, K, N in LINEARS_70B])


@pytest.mark.parametrize("name,M,N,K,scaling,transposes,micro_batches", FULL_CASES,
                         ids=[c[0] for c in FULL_CASES])
def test_full_size_linear_sampled(name, M, N, K, scaling, transposes, micro_batches):
    """Every linear of the two transformer blocks at full size, with the
    oracle's own state machine: X, W and dY codes and all scales bit-exact;
    64 seeded rows and 64 seeded full columns of each of Y, dX and dW within
    the GEMM bound.  The Llama-2-70B cases accumulate dW over two
    micro-batches (the second checked against the first's dW plus the
    oracle's second product)."""
    recipe = (F.Recipe(F.SCALING_DELAYED, history_len=16) if scaling == F.SCALING_DELAYED
              else F.Recipe(F.SCALING_DYNAMIC))
    layer = F.Fp8Linear(M, N, K, recipe, device=DEV, transposes=transposes)
    orec = _orecipe(recipe)
    ost = oracle.LinearState(orec)
    W = synthetic.normal((N, K), 0.02, seed=2, device=DEV)
    bw = bits(W)
    dW = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    rows_m, cols_n = _sample(M, SAMPLE, 1), _sample(N, SAMPLE, 2)
    rows_n, cols_k = _sample(N, SAMPLE, 3), _sample(K, SAMPLE, 4)
    tm, tn, tk = (torch.as_tensor(v, device=DEV) for v in (rows_m, rows_n, cols_k))
    tcn = torch.as_tensor(cols_n, device=DEV)
    prev_r = prev_c = None
    for mb in range(micro_batches):
        X = synthetic.with_outlier_channels((M, K), 1.0, _outlier_channels(K), 50.0,
                                            seed=10 + mb, device=DEV)
        dY = synthetic.normal((M, N), 1e-3, seed=20 + mb, device=DEV)
        Y = layer.forward(X, W)
        dX, _ = layer.backward(dY, dW=dW, accumulate_dW=mb > 0)
        torch.cuda.synchronize()
        Yo, Yabs = oracle.linear_fwd(bits(X), bw, orec, ost, rows=rows_m)
        (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost, rows_dx=rows_m,
                                                       rows_dw=rows_n)
        # the quantised operands (dY's codes live in the workspace) and every scale
        assert np.array_equal(u8(layer.x_q), ost.x_q)
        assert np.array_equal(u8(layer.w_q), ost.w_q)
        assert np.array_equal(u8(layer.workspace[:M * N]).reshape(M, N), ost.dy_q)
        if transposes:
            assert np.array_equal(u8(layer.x_qt), ost.x_qt)
            assert np.array_equal(u8(layer.w_qt), ost.w_qt)
        _check_state(layer, ost)
        sx, sw = ost.sinv_fwd
        sdy = ost.sinv_bwd
        Yc, Ycabs = _columns(ost.x_q, F.E4M3, ost.w_q, F.E4M3, sx, sw, M, cols_n)
        dXc, dXcabs = _columns(ost.dy_q, F.E5M2, ost.w_qt, F.E4M3, sdy, sw, M, cols_k)
        dWc, dWcabs = _columns(ost.dy_qt, F.E5M2, ost.x_qt, F.E4M3, sdy, sx, N, cols_k)
        what = f"{name}, micro-batch {mb}"
        assert_gemm_bound(Y[tm], Yo, Yabs, what=what + " Y rows")
        assert_gemm_bound(Y[:, tcn], Yc, Ycabs, what=what + " Y columns")
        assert_gemm_bound(dX[tm], dXo, dXabs, what=what + " dX rows")
        assert_gemm_bound(dX[:, tk], dXc, dXcabs, what=what + " dX columns")
        if prev_r is None:
            assert_gemm_bound(dW[tn], dWo, dWabs, what=what + " dW rows")
            assert_gemm_bound(dW[:, tk], dWc, dWcabs, what=what + " dW columns")
        else:
            assert_gemm_bound(dW[tn], dWo + prev_r, dWabs, prev=prev_r, what=what + " dW rows")
            assert_gemm_bound(dW[:, tk], dWc + prev_c, dWcabs, prev=prev_c,
                              what=what + " dW columns")
        prev_r = dW[tn].cpu().numpy().astype(np.float64)
        prev_c = dW[:, tk].cpu().numpy().astype(np.float64)


BLOCK_SAMPLE = 32


@pytest.mark.parametrize("M,N,K", [(16384, 18432, 7168), (16384, 7168, 18432)])
@pytest.mark.parametrize("pow2", [False, True], ids=["fp32_scales", "pow2_scales"])
def test_full_size_block_layer_sampled(M, N, K, pow2):
    """The block-wise layer (1x128 activations and gradients, 128x128
    weights) forward and backward at the DeepSeek-style shapes: every code
    and block scale of X, X^T, W, W^T, dY and dY^T bit-exact against the
    oracle's casts; 32 seeded rows and 32 full columns of Y, dX and dW within
    the GEMM bound."""
    rec = F.Recipe(F.SCALING_BLOCK, pow2=pow2)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    X = synthetic.student_t_rows((M, K), 1.0, 3, seed=11, device=DEV)
    W = synthetic.student_t_rows((N, K), 0.02, 3, seed=12, device=DEV)
    dY = synthetic.normal((M, N), 1e-3, seed=13, device=DEV)
    Y = layer.forward(X, W)
    dX, dW = layer.backward(dY)
    torch.cuda.synchronize()
    orec = _orecipe(rec)
    ost = oracle.LinearState(orec)
    rows_m, cols_n = _sample(M, BLOCK_SAMPLE, 5), _sample(N, BLOCK_SAMPLE, 6)
    rows_n, cols_k = _sample(N, BLOCK_SAMPLE, 7), _sample(K, BLOCK_SAMPLE, 8)
    Yo, Yabs = oracle.linear_fwd(bits(X), bits(W), orec, ost, rows=rows_m)
    (dXo, dXabs), (dWo, dWabs) = oracle.linear_bwd(bits(dY), orec, ost, rows_dx=rows_m,
                                                   rows_dw=rows_n)
    for got, want in ((layer.x_q, ost.x_q), (layer.x_qt, ost.xt_q), (layer.w_q, ost.w_q),
                      (layer.w_qt, ost.wt_q)):
        assert np.array_equal(u8(got), want)
    for got, want in ((layer.x_sinv, ost.x_sinv), (layer.x_sinv_t, ost.xt_sinv),
                      (layer.w_sinv, ost.w_sinv), (layer.w_sinv_t, ost.wt_sinv)):
        assert np.array_equal(f32bits(got.cpu().numpy()), f32bits(want))
    _check_block_dy(layer, ost, M, N)
    G1, G2 = oracle.GRAN_1x128, oracle.GRAN_128x128
    Yc, Ycabs = _columns(ost.x_q, F.E4M3, ost.w_q, F.E4M3, ost.x_sinv, ost.w_sinv, M, cols_n,
                         G1, G2)
    dXc, dXcabs = _columns(ost.dy_q, F.E5M2, ost.wt_q, F.E4M3, ost.dy_s, ost.wt_sinv, M, cols_k,
                           G1, G2)
    dWc, dWcabs = _columns(ost.dyt_q, F.E5M2, ost.xt_q, F.E4M3, ost.dyt_s, ost.xt_sinv, N,
                           cols_k, G1, G1)
    tm, tn, tk = (torch.as_tensor(v, device=DEV) for v in (rows_m, rows_n, cols_k))
    assert_gemm_bound(Y[tm], Yo, Yabs, what="Y rows")
    assert_gemm_bound(Y[:, torch.as_tensor(cols_n, device=DEV)], Yc, Ycabs, what="Y columns")
    assert_gemm_bound(dX[tm], dXo, dXabs, what="dX rows")
    assert_gemm_bound(dX[:, tk], dXc, dXcabs, what="dX columns")
    assert_gemm_bound(dW[tn], dWo, dWabs, what="dW rows")
    assert_gemm_bound(dW[:, tk], dWc, dWcabs, what="dW columns")


def test_step_replays_from_a_cuda_graph():
    """fp8_linear_fwd + fp8_linear_bwd captured once in a CUDA graph and
    replayed: every output bit equal to the eager calls on the same state
    (dynamic scaling, so the state does not drift between the runs)."""
    M, N, K = 256, 512, 512
    dev = torch.device(DEV)
    rec = F.Recipe(F.SCALING_DYNAMIC)
    eager = F.Fp8Linear(M, N, K, rec, device=DEV)
    graphed = F.Fp8Linear(M, N, K, rec, device=DEV)
    X = synthetic.with_outlier_entries((M, K), 1.0, 0.001, 50.0, seed=0).to(dev)
    W = synthetic.normal((N, K), 0.02, seed=1).to(dev)
    dY = synthetic.normal((M, N), 1e-3, seed=2).to(dev)
    b = synthetic.normal((N,), 0.1, seed=3).to(dev)
    outs = {}
    for name, layer in (("eager", eager), ("graph", graphed)):
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dW = torch.zeros(N, K, dtype=torch.float32, device=dev)
        db = torch.zeros(N, dtype=torch.float32, device=dev)

        def run():
            layer.forward(X, W, Y=Y, bias=b)
            layer.backward(dY, dX=dX, dW=dW, dbias=db)
        if name == "eager":
            run()
        else:
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                run()                                # warm-up outside the capture
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    run()
            torch.cuda.current_stream().wait_stream(side)
            for t in (Y, dX, dW, db):
                t.zero_()
            g.replay()
            g.replay()
        torch.cuda.synchronize()
        outs[name] = [t.clone() for t in (Y, dX, dW, db)]
    for a, c in zip(outs["eager"], outs["graph"]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           c.view(torch.int16) if c.dtype == torch.bfloat16 else c.view(torch.int32))


@pytest.mark.parametrize("transposes", [False, True], ids=["fused_update", "update_kernel"])
def test_dynamic_non_finite_and_zero_inputs(transposes):
    """Dynamic scaling (the scale computed inside the cast when no transposed
    copies are kept, by the update kernel otherwise): a NaN in X keeps the X
    scale and sets bit 1 of the device status word for that step only; an
    all-zero dY keeps the dY scale; every other role and step matches the
    oracle's state machine bit for bit."""
    M, N, K = 256, 256, 256
    rec = F.Recipe(F.SCALING_DYNAMIC)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV, transposes=transposes)
    ost = oracle.LinearState(_orecipe(rec))
    W = synthetic.normal((N, K), 0.02, seed=1)
    flags = []
    for step in range(4):
        X = synthetic.normal((M, K), 1.0, seed=10 + step)
        dY = synthetic.normal((M, N), 1e-3, seed=20 + step)
        if step == 1:
            X[5, 7] = float("nan")
        if step == 2:
            dY.zero_()
        before = layer.scale.clone()
        layer.forward(X.to(DEV), W.to(DEV))
        layer.backward(dY.to(DEV))
        flags.append(F.fp8_device_status(clear=True))
        oracle.linear_fwd(bits(X), bits(W), _orecipe(rec), ost)
        oracle.linear_bwd(bits(dY), _orecipe(rec), ost)
        if step == 1:
            assert layer.scale[0].item() == before[0].item()
        if step == 2:
            assert layer.scale[2].item() == before[2].item()
        _check_state(layer, ost)
    assert flags == [0, 2, 0, 0]


def test_non_finite_input_is_flagged_and_the_scale_held():
    """A NaN in X: the delayed update keeps the X scale and sets bit 1 of the
    device status word, at this step and for as long as the NaN stays in the
    amax history (4 steps here); the other roles are unaffected."""
    M, N, K = 256, 256, 256
    rec = F.Recipe(F.SCALING_DELAYED, history_len=4)
    layer = F.Fp8Linear(M, N, K, rec, device=DEV)
    W = synthetic.normal((N, K), 0.02, seed=1).to(DEV)
    flags = []
    for step in range(7):
        X = synthetic.normal((M, K), 1.0, seed=10 + step)
        if step == 1:
            X[5, 7] = float("nan")
        before = layer.scale.clone()
        layer.forward(X.to(DEV), W)
        flags.append(F.fp8_device_status(clear=True))
        if step >= 1 and step <= 4:
            assert layer.scale[0].item() == before[0].item(), step
    assert flags == [0, 2, 2, 2, 2, 0, 0]
