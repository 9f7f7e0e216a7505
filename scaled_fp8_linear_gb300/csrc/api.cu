// api.cu -- the extern "C" boundary (include/fp8linear.h): argument checks,
// the composition of the linear layer's forward and backward passes out of
// the quantiser and GEMM launchers, and error reporting.
//
// Forward / backward composition ("Mixed Precision LLM Training: The
// Complete Guide", "Transformer Engine internals" > "Delayed scaling" and
// "The HYBRID recipe"; "FP8 and gradient accumulation"):
//   fwd delayed:  q(X), q(W) with the current scales, fused amax + transpose
//                 -> GEMM -> scale update of X and W (used from the next call)
//   fwd dynamic:  amax(X), amax(W) -> scale update -> q(X), q(W) -> GEMM
//   fwd block:    1x128 q(X), 128x128 q(W) -> block-scaled GEMM
//   bwd:          q(dY) (E5M2) + transpose -> dgrad GEMM dY . W
//                 -> wgrad GEMM dY^T . X into the FP32 buffer -> dY scale update
// Every step is one kernel launch on the caller's stream; nothing waits on
// the host.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fp8linear.h"
#include "internal.h"

namespace fp8 {

namespace {
thread_local std::string g_last_error;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId, through the runtime's entry
// point query (null when the driver lacks them).
std::pair<CtxGetCurrentFn, CtxGetIdFn> ctx_fns() {
    static CtxGetCurrentFn cur = nullptr;
    static CtxGetIdFn id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return {cur, id};
}

// Unique ID of the calling thread's current CUDA context, 0 if there is none
// (or it cannot be read).  The driver never reuses an ID within a process,
// so a context made after cudaDeviceReset, or another context made current
// by the caller, has an ID of its own.
unsigned long long current_context_id_impl() {
    const auto fns = ctx_fns();
    if (!fns.first || !fns.second) return 0;
    CUcontext ctx = nullptr;
    if (fns.first(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (fns.second(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

unsigned long long current_context_id() { return current_context_id_impl(); }

int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_format(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
bool valid_gran(int g) { return g >= FP8_GRAN_TENSOR && g <= FP8_GRAN_ROW; }
bool block_gran(int g) { return g == FP8_GRAN_1x128 || g == FP8_GRAN_128x128; }
// A GEMM operand's granularity: a valid one, with FP8_SCALE_POW2 only on
// block granularities.
bool valid_gemm_gran(int g) {
    const int base = g & ~FP8_SCALE_POW2;
    return valid_gran(base) && (!(g & FP8_SCALE_POW2) || block_gran(base));
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FP8_OK;
    return set_error(FP8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define FP8_CHECK(expr)                  \
    do {                                 \
        const int st_ = (expr);          \
        if (st_ != FP8_OK) return st_;   \
    } while (0)

int check_recipe(const fp8_recipe_t* r) {
    if (!r) return set_error(FP8_ERR_INVALID_ARG, "recipe is NULL");
    if (r->scaling < FP8_SCALING_DELAYED || r->scaling > FP8_SCALING_ROW)
        return set_error(FP8_ERR_INVALID_ARG, "unknown scaling mode %d", r->scaling);
    if (r->margin < 0 || r->margin > 64)
        return set_error(FP8_ERR_INVALID_ARG, "margin %d outside 0..64", r->margin);
    if (r->scaling == FP8_SCALING_DELAYED && (r->history_len < 1 || r->history_len > 1024))
        return set_error(FP8_ERR_INVALID_ARG, "history_len %d outside 1..1024", r->history_len);
    if (r->amax_algo != FP8_AMAX_MAX && r->amax_algo != FP8_AMAX_MOST_RECENT)
        return set_error(FP8_ERR_INVALID_ARG, "unknown amax_algo %d", r->amax_algo);
    if (!valid_format(r->fwd_format) || !valid_format(r->bwd_format))
        return set_error(FP8_ERR_INVALID_ARG, "unknown FP8 format");
    if (r->sr_grad != 0 && r->sr_grad != 1)
        return set_error(FP8_ERR_INVALID_ARG, "sr_grad %d is not 0 or 1", r->sr_grad);
    if (r->sr_grad && (r->scaling == FP8_SCALING_BLOCK || r->scaling == FP8_SCALING_ROW))
        return set_error(FP8_ERR_UNSUPPORTED,
                         "sr_grad: stochastic rounding of dY is built for per-tensor scaling only");
    return FP8_OK;
}

int history_len_of(const fp8_recipe_t* r) {
    return r->scaling == FP8_SCALING_DELAYED ? r->history_len : 1;
}

int check_gemm_args(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                    int64_t K, int layout, int ga, const float* sa, int gb, const float* sb,
                    const void* D, int out, int accumulate) {
    if (!sa || !sb) return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: NULL scale pointer");
    if ((!A && M > 0 && K > 0) || (!B && N > 0 && K > 0) || (!D && M > 0 && N > 0))
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: NULL pointer");
    if (!valid_format(fa) || !valid_format(fb))
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: unknown FP8 format");
    if (layout < FP8_LAYOUT_TN || layout > FP8_LAYOUT_KM_KN)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: unknown layout %d", layout);
    if (!valid_gemm_gran(ga) || !valid_gemm_gran(gb))
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: unknown scale granularity");
    ga &= ~FP8_SCALE_POW2;
    gb &= ~FP8_SCALE_POW2;
    if (out != FP8_OUT_BF16 && out != FP8_OUT_F32)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: unknown output type %d", out);
    if (accumulate && out != FP8_OUT_F32)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm: accumulate needs FP32 output");
    if (M < 0 || N < 0 || K < 0 || M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31))
        return set_error(FP8_ERR_SHAPE, "fp8_gemm: dimensions out of range");
    if (N % 16 || K % 16) return set_error(FP8_ERR_SHAPE, "fp8_gemm: N and K must be multiples of 16");
    const bool block = block_gran(ga) || block_gran(gb);
    if (block && (ga == FP8_GRAN_ROW || gb == FP8_GRAN_ROW))
        return set_error(FP8_ERR_UNSUPPORTED, "fp8_gemm: per-row and block scales cannot be mixed");
    if (block && layout != FP8_LAYOUT_TN)
        return set_error(FP8_ERR_UNSUPPORTED, "fp8_gemm: block scales need layout FP8_LAYOUT_TN");
    if ((layout & FP8_LAYOUT_A_KM) && M % 16)
        return set_error(FP8_ERR_SHAPE, "fp8_gemm: A stored [K x M] needs M multiple of 16");
    if (block) {
        if (K % 128 || N % 128)
            return set_error(FP8_ERR_SHAPE, "fp8_gemm: block scales need N and K multiples of 128");
        if (ga == FP8_GRAN_128x128 && M % 128)
            return set_error(FP8_ERR_SHAPE, "fp8_gemm: 128x128 scales on A need M multiple of 128");
    }
    if (!aligned16(A) || !aligned16(B) || !aligned16(D))
        return set_error(FP8_ERR_ALIGN, "fp8_gemm: A, B and D must be 16-byte aligned");
    return FP8_OK;
}

int check_quantize_args(const void* x, int64_t rows, int64_t cols, int format, int gran,
                        const float* scale, uint8_t* q, uint8_t* q_t, float* sinv, float* sinv_t,
                        float* amax_out) {
    if ((!x || !q) && rows > 0 && cols > 0)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: NULL pointer");
    if (!valid_format(format)) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: unknown format");
    if (!valid_gran(gran)) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: unknown granularity");
    if (rows < 0 || cols < 0) return set_error(FP8_ERR_SHAPE, "fp8_quantize: negative dimension");
    if (gran == FP8_GRAN_TENSOR) {
        if (!scale) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: scale is NULL");
        if (q_t && (rows % 16 || cols % 16))
            return set_error(FP8_ERR_SHAPE, "fp8_quantize: the transpose needs rows and cols multiples of 16");
    } else if (gran == FP8_GRAN_ROW) {
        if (!sinv) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: scale_inv_blocks is NULL");
        if (amax_out || scale)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: per-row mode takes no scale or amax_out");
        if (q_t && !sinv_t)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: q_t needs scale_inv_blocks_t in per-row mode");
        if (cols % 16 || (q_t && rows % 16))
            return set_error(FP8_ERR_SHAPE, "fp8_quantize: per-row mode needs cols (and, with q_t, rows) multiples of 16");
    } else {
        if (!sinv) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: scale_inv_blocks is NULL");
        if (amax_out || scale)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: block modes take no scale or amax_out");
        if (q_t && !sinv_t)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize: q_t needs scale_inv_blocks_t in block modes");
        if (cols % 128) return set_error(FP8_ERR_SHAPE, "fp8_quantize: block modes need cols multiple of 128");
        if ((gran == FP8_GRAN_128x128 || q_t) && rows % 128)
            return set_error(FP8_ERR_SHAPE, "fp8_quantize: 128x128 blocks and block transposes need rows multiple of 128");
    }
    if (!aligned16(x) || !aligned16(q) || (q_t && !aligned16(q_t)))
        return set_error(FP8_ERR_ALIGN, "fp8_quantize: x, q and q_t must be 16-byte aligned");
    return FP8_OK;
}

int check_linear_shape(int64_t M, int64_t N, int64_t K, const fp8_recipe_t* r) {
    if (M < 0 || N < 0 || K < 0 || M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31))
        return set_error(FP8_ERR_SHAPE, "linear: dimensions out of range");
    const int64_t mult = r->scaling == FP8_SCALING_BLOCK ? 128 : 16;
    if (N % mult || K % mult || (r->scaling != FP8_SCALING_BLOCK && M % mult))
        return set_error(FP8_ERR_SHAPE, "linear: M, N, K must be multiples of %lld", (long long)mult);
    return FP8_OK;
}

int check_state_scales(const fp8_linear_state_t* s) {
    if (!s) return set_error(FP8_ERR_INVALID_ARG, "linear: state is NULL");
    if (!s->scale || !s->scale_inv || !s->amax || !s->history || !s->pos || !s->qscale_inv)
        return set_error(FP8_ERR_INVALID_ARG, "linear: state scale arrays must be set");
    return FP8_OK;
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Workspace of the backward pass, in order: the dY operands (dY_q, dY_q^T,
// and their scale arrays in the block-wise and per-row modes), then the bias
// gradient's partial column sums, one row of N floats per 128 tokens.
// With a state (s non-null) the per-tensor modes count what that state's
// backward writes: dY_q alone when the forward kept no transposed copies
// (the GEMMs then read the codes MN-major), dY_q and dY_q^T otherwise.
size_t bwd_operand_bytes(int64_t M, int64_t N, const fp8_recipe_t* recipe,
                         const fp8_linear_state_t* s = nullptr) {
    const size_t mn = static_cast<size_t>(M) * static_cast<size_t>(N);
    if (recipe->scaling == FP8_SCALING_ROW)   // + per-row scales of both, [M] and [N]
        return 2 * align256(mn) + align256(4 * static_cast<size_t>(M)) +
               align256(4 * static_cast<size_t>(N));
    if (recipe->scaling == FP8_SCALING_BLOCK)  // + 1x128 scales, [M][N/128] and [N][M/128]
        return 2 * align256(mn) + 2 * align256(4 * (mn / 128));
    if (s && !(s->x_qt && s->w_qt)) return align256(mn);
    return 2 * align256(mn);
}

size_t dbias_partial_bytes(int64_t M, int64_t N) {
    return align256(4 * static_cast<size_t>((M + 127) / 128) * static_cast<size_t>(N));
}

// The dynamic update of role r (its history has length 1), for a cast that
// fuses it.
ScaleUpd dynamic_update(const fp8_linear_state_t* s, int r, const fp8_recipe_t* recipe,
                        float* saved) {
    return ScaleUpd{s->amax + r, s->history + r, s->pos + r, recipe->margin, recipe->pow2 != 0,
                    s->scale + r, s->scale_inv + r, saved, device_status_word()};
}

// The forward's per-tensor casts of X and W (with their amax if `amax`):
// one launch over both tensors when both transposes or neither are kept,
// else one cast each.
cudaError_t quantize_x_w(const void* X, const void* W, int64_t M, int64_t N, int64_t K, int f,
                         const fp8_linear_state_t* s, bool amax, cudaStream_t st) {
    if ((s->x_qt && s->w_qt) || (!s->x_qt && !s->w_qt))
        return launch_quantize_pair(X, M, K, s->scale + 0, s->x_q, s->x_qt, amax ? s->amax + 0 : nullptr,
                                    W, N, K, s->scale + 1, s->w_q, s->w_qt, amax ? s->amax + 1 : nullptr,
                                    f, st);
    cudaError_t e = launch_quantize_tensor(X, M, K, f, s->scale + 0, s->x_q, s->x_qt,
                                           amax ? s->amax + 0 : nullptr, st);
    if (e != cudaSuccess) return e;
    return launch_quantize_tensor(W, N, K, f, s->scale + 1, s->w_q, s->w_qt,
                                  amax ? s->amax + 1 : nullptr, st);
}

// The workspace of a backward call: its size (the partial sums only when
// dbias is wanted) and alignment.
int check_bwd_workspace(int64_t M, int64_t N, const fp8_recipe_t* recipe,
                        const fp8_linear_state_t* s, const float* dbias, const void* workspace,
                        size_t workspace_bytes) {
    const size_t need = bwd_operand_bytes(M, N, recipe, s) + (dbias ? dbias_partial_bytes(M, N) : 0);
    if (!workspace && need) return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_bwd: NULL pointer");
    if (workspace_bytes < need)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_bwd: workspace of %zu bytes, %zu needed",
                         workspace_bytes, need);
    if (!aligned16(workspace))
        return set_error(FP8_ERR_ALIGN, "fp8_linear_bwd: tensors must be 16-byte aligned (dbias 4-byte)");
    return FP8_OK;
}

// Block-wise backward ("DeepSeek FP8 training recipe" > "Block-wise scaling
// at 128 granularity"): one dual cast of dY gives the dgrad operand (1x128
// blocks along N) and the wgrad operand (dY^T, 1x128 blocks along the
// tokens); dgrad uses W_q^T with its 128x128 scales, wgrad X^T's 1x128
// token-blocked cast kept by the forward pass.
int linear_bwd_block(const void* dY, int64_t M, int64_t N, int64_t K, const fp8_recipe_t* recipe,
                     const fp8_linear_state_t* s, void* dX, float* dW, int accumulate_dW,
                     float* dbias, void* workspace, cudaStream_t st) {
    const size_t mn = static_cast<size_t>(M) * static_cast<size_t>(N);
    const int fb = recipe->bwd_format, ff = recipe->fwd_format;
    uint8_t* dy_q = static_cast<uint8_t*>(workspace);
    uint8_t* dy_qt = dy_q + align256(mn);
    float* dy_s = reinterpret_cast<float*>(dy_qt + align256(mn));
    float* dy_st = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dy_s) + align256(4 * (mn / 128)));
    FP8_CHECK(cuda_status(launch_quantize_block(dY, M, N, fb, FP8_GRAN_1x128, recipe->pow2 != 0,
                                                dy_q, dy_s, dy_qt, dy_st, st), "quantize dY"));
    if (dbias) {
        float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                  bwd_operand_bytes(M, N, recipe));
        FP8_CHECK(cuda_status(launch_dbias(dY, M, N, partial, false, dbias, accumulate_dW, st),
                              "dbias"));
    }
    // power-of-two factors (pow2 casts) go to the block-scaled MMA
    const int p2 = recipe->pow2 ? FP8_SCALE_POW2 : 0;
    // dgrad: dX [M x K] = dY_q [M x N] . (W_q^T [K x N])^T
    FP8_CHECK(launch_gemm(dy_q, fb, s->w_qt, ff, M, K, N, FP8_GRAN_1x128 | p2, dy_s,
                          FP8_GRAN_128x128 | p2, s->w_sinv_t, nullptr, dX, FP8_OUT_BF16, 0, st));
    // wgrad: dW [N x K] (+)= dY_q^T [N x M] . (X_q^T [K x M])^T
    return launch_gemm(dy_qt, fb, s->x_qt, ff, N, K, M, FP8_GRAN_1x128 | p2, dy_st,
                       FP8_GRAN_1x128 | p2, s->x_sinv_t, nullptr, dW, FP8_OUT_F32,
                       accumulate_dW != 0, st);
}

// Per-row backward: dY cast per token (dgrad operand) and per output
// channel (dY^T, wgrad operand); dgrad takes W^T's per-input-channel cast
// and wgrad X^T's, both kept by the forward pass.  Every factor is per row
// or per column of the GEMM output, so all three GEMMs are per-tensor-kernel
// GEMMs with vector epilogue factors.
int linear_bwd_row(const void* dY, int64_t M, int64_t N, int64_t K, const fp8_recipe_t* recipe,
                   const fp8_linear_state_t* s, void* dX, float* dW, int accumulate_dW,
                   float* dbias, void* workspace, cudaStream_t st) {
    const size_t mn = static_cast<size_t>(M) * static_cast<size_t>(N);
    const int fb = recipe->bwd_format, ff = recipe->fwd_format;
    uint8_t* dy_q = static_cast<uint8_t*>(workspace);
    uint8_t* dy_qt = dy_q + align256(mn);
    float* dy_s = reinterpret_cast<float*>(dy_qt + align256(mn));
    float* dy_st = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dy_s) + align256(4 * static_cast<size_t>(M)));
    FP8_CHECK(cuda_status(launch_quantize_rows(dY, M, N, fb, recipe->pow2 != 0, dy_q, dy_s, dy_qt,
                                               dy_st, st), "quantize dY"));
    if (dbias) {
        float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                  bwd_operand_bytes(M, N, recipe));
        FP8_CHECK(cuda_status(launch_dbias(dY, M, N, partial, false, dbias, accumulate_dW, st),
                              "dbias"));
    }
    return launch_gemm_group(
        GemmArgs{dy_q, fb, s->w_qt, ff, M, K, N, FP8_GRAN_ROW, dy_s, FP8_GRAN_ROW, s->w_sinv_t,
                 nullptr, dX, FP8_OUT_BF16, 0},
        GemmArgs{dy_qt, fb, s->x_qt, ff, N, K, M, FP8_GRAN_ROW, dy_st, FP8_GRAN_ROW, s->x_sinv_t,
                 nullptr, dW, FP8_OUT_F32, accumulate_dW != 0},
        st);
}

}  // namespace

int check_linear_bwd_args(const void* dY, int64_t M, int64_t N, int64_t K,
                          const fp8_recipe_t* recipe, const fp8_linear_state_t* s, const void* dX,
                          const float* dW, const float* dbias) {
    FP8_CHECK(check_recipe(recipe));
    FP8_CHECK(check_linear_shape(M, N, K, recipe));
    // M = 0: dY, dX and the forward's M-sized operands may be NULL; dW (and
    // dbias) are written (zero) or, with accumulate_dW, left as they are
    if ((!dY && M) || (!dX && M) || !dW || !s)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_bwd: NULL pointer");
    const bool block = recipe->scaling == FP8_SCALING_BLOCK;
    if (block || recipe->scaling == FP8_SCALING_ROW) {
        if (M && (!s->x_qt || !s->w_qt || !s->x_sinv_t || !s->w_sinv_t))
            return set_error(FP8_ERR_INVALID_ARG,
                             "fp8_linear_bwd: %s mode needs the forward's x_qt/x_sinv_t and w_qt/w_sinv_t",
                             block ? "block" : "per-row");
        if (block && M % 128)
            return set_error(FP8_ERR_SHAPE, "fp8_linear_bwd: block mode needs M multiple of 128");
    } else {
        FP8_CHECK(check_state_scales(s));
        if ((!s->x_q && M) || !s->w_q)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_bwd: state->x_q / w_q must be set");
        if (recipe->sr_grad && (!s->sr_key || (reinterpret_cast<uintptr_t>(s->sr_key) & 7u)))
            return set_error(FP8_ERR_INVALID_ARG,
                             "fp8_linear_bwd: sr_grad needs an 8-byte aligned state->sr_key");
    }
    if (!aligned16(dY) || !aligned16(dX) || !aligned16(dW) || !aligned16(s->x_q) ||
        !aligned16(s->w_q) || !aligned16(s->x_qt) || !aligned16(s->w_qt) ||
        (reinterpret_cast<uintptr_t>(dbias) & 3u))
        return set_error(FP8_ERR_ALIGN, "fp8_linear_bwd: tensors must be 16-byte aligned (dbias 4-byte)");
    return FP8_OK;
}

size_t bwd_operand_workspace(int64_t M, int64_t N, const fp8_recipe_t* recipe,
                             const fp8_linear_state_t* s) {
    return bwd_operand_bytes(M, N, recipe, s);
}

}  // namespace fp8

using namespace fp8;

extern "C" {

const char* fp8_last_error(void) { return g_last_error.c_str(); }

int fp8_amax(const void* x, int64_t n, float* amax, void* stream) {
    if (!amax || (!x && n > 0)) return set_error(FP8_ERR_INVALID_ARG, "fp8_amax: NULL pointer");
    if (n < 0) return set_error(FP8_ERR_SHAPE, "fp8_amax: negative size");
    if (!aligned16(x)) return set_error(FP8_ERR_ALIGN, "fp8_amax: x must be 16-byte aligned");
    return cuda_status(launch_amax(x, n, amax, as_stream(stream)), "fp8_amax");
}

int fp8_update_scale(const float* amax, float* history, int32_t* pos, int history_len, int algo,
                     int format, int margin, int pow2, float* scale, float* scale_inv,
                     void* stream) {
    if (!amax || !history || !pos || !scale || !scale_inv)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_update_scale: NULL pointer");
    if (history_len < 1 || history_len > 1024)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_update_scale: history_len %d outside 1..1024", history_len);
    if (algo != FP8_AMAX_MAX && algo != FP8_AMAX_MOST_RECENT)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_update_scale: unknown algo %d", algo);
    if (!valid_format(format)) return set_error(FP8_ERR_INVALID_ARG, "fp8_update_scale: unknown format");
    if (margin < 0 || margin > 64)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_update_scale: margin %d outside 0..64", margin);
    return cuda_status(launch_update_scale(amax, history, pos, history_len, algo, format, margin,
                                           pow2 != 0, scale, scale_inv, 1, as_stream(stream)),
                       "fp8_update_scale");
}

int fp8_quantize(const void* x, int64_t rows, int64_t cols, int format, int granularity,
                 const float* scale, int pow2, uint8_t* q, uint8_t* q_t, float* scale_inv_blocks,
                 float* scale_inv_blocks_t, float* amax_out, void* stream) {
    FP8_CHECK(check_quantize_args(x, rows, cols, format, granularity, scale, q, q_t,
                                  scale_inv_blocks, scale_inv_blocks_t, amax_out));
    if (granularity == FP8_GRAN_TENSOR)
        return cuda_status(launch_quantize_tensor(x, rows, cols, format, scale, q, q_t, amax_out,
                                                  as_stream(stream)),
                           "fp8_quantize");
    if (granularity == FP8_GRAN_ROW)
        return cuda_status(launch_quantize_rows(x, rows, cols, format, pow2 != 0, q,
                                                scale_inv_blocks, q_t, scale_inv_blocks_t,
                                                as_stream(stream)),
                           "fp8_quantize");
    return cuda_status(launch_quantize_block(x, rows, cols, format, granularity, pow2 != 0, q,
                                             scale_inv_blocks, q_t, scale_inv_blocks_t,
                                             as_stream(stream)),
                       "fp8_quantize");
}

int fp8_quantize_counted(const void* x, int64_t rows, int64_t cols, int format,
                         const float* scale, uint8_t* q, uint8_t* q_t, float* amax_out,
                         unsigned long long* counts, void* stream) {
    FP8_CHECK(check_quantize_args(x, rows, cols, format, FP8_GRAN_TENSOR, scale, q, q_t, nullptr,
                                  nullptr, amax_out));
    if (!counts) return set_error(FP8_ERR_INVALID_ARG, "fp8_quantize_counted: counts is NULL");
    if (reinterpret_cast<uintptr_t>(counts) & 7u)
        return set_error(FP8_ERR_ALIGN, "fp8_quantize_counted: counts must be 8-byte aligned");
    return cuda_status(launch_quantize_tensor(x, rows, cols, format, scale, q, q_t, amax_out,
                                              as_stream(stream), counts),
                       "fp8_quantize_counted");
}

int fp8_quantize_sr(const void* x, int64_t rows, int64_t cols, int format, const float* scale,
                    uint64_t seed, uint64_t offset, uint8_t* q, uint8_t* q_t, float* amax_out,
                    void* stream) {
    FP8_CHECK(check_quantize_args(x, rows, cols, format, FP8_GRAN_TENSOR, scale, q, q_t, nullptr,
                                  nullptr, amax_out));
    return cuda_status(launch_quantize_sr(x, rows, cols, format, scale, seed, offset, q, q_t,
                                          amax_out, as_stream(stream)),
                       "fp8_quantize_sr");
}

int fp8_gemm(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N, int64_t K,
             int layout, int ga, const float* scale_inv_a, int gb, const float* scale_inv_b,
             const void* bias, void* D, int out, int accumulate, void* stream) {
    FP8_CHECK(check_gemm_args(A, fa, B, fb, M, N, K, layout, ga, scale_inv_a, gb, scale_inv_b, D,
                              out, accumulate));
    if (bias && !aligned16(bias))
        return set_error(FP8_ERR_ALIGN, "fp8_gemm: bias must be 16-byte aligned");
    return launch_gemm(A, fa, B, fb, M, N, K, ga, scale_inv_a, gb, scale_inv_b, bias, D, out,
                       accumulate != 0, as_stream(stream), layout);
}

int fp8_gemm_group(const fp8_gemm_args_t* g1, const fp8_gemm_args_t* g2, void* stream) {
    if (!g1 || !g2) return set_error(FP8_ERR_INVALID_ARG, "fp8_gemm_group: NULL problem");
    for (const fp8_gemm_args_t* g : {g1, g2}) {
        FP8_CHECK(check_gemm_args(g->A, g->fa, g->B, g->fb, g->M, g->N, g->K, g->layout, g->ga,
                                  g->scale_inv_a, g->gb, g->scale_inv_b, g->D, g->out,
                                  g->accumulate));
        if (g->bias && !aligned16(g->bias))
            return set_error(FP8_ERR_ALIGN, "fp8_gemm_group: bias must be 16-byte aligned");
    }
    auto args = [](const fp8_gemm_args_t* g) {
        return GemmArgs{g->A, g->fa, g->B, g->fb, g->M, g->N, g->K, g->ga, g->scale_inv_a,
                        g->gb, g->scale_inv_b, g->bias, g->D, g->out, g->accumulate != 0,
                        g->layout};
    };
    return launch_gemm_group(args(g1), args(g2), as_stream(stream));
}

size_t fp8_workspace_size(int64_t M, int64_t N, int64_t K, const fp8_recipe_t* recipe) {
    (void)K;
    if (check_recipe(recipe) != FP8_OK || M < 0 || N < 0) return 0;
    return bwd_operand_bytes(M, N, recipe) + dbias_partial_bytes(M, N);
}

int fp8_linear_fwd(const void* X, const void* W, const void* bias, int64_t M, int64_t N,
                   int64_t K, const fp8_recipe_t* recipe, const fp8_linear_state_t* s, void* Y,
                   void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    FP8_CHECK(check_recipe(recipe));
    FP8_CHECK(check_linear_shape(M, N, K, recipe));
    // M = 0 (a batch without tokens): the M-sized buffers X, Y, x_q, x_qt and
    // x_sinv may be NULL
    if ((!X && M) || !W || (!Y && M) || !s)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: NULL pointer");
    if ((!s->x_q && M) || !s->w_q)
        return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: state->x_q / w_q must be set");
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(s->x_q) || !aligned16(s->w_q) ||
        (bias && !aligned16(bias)) ||
        (s->x_qt && !aligned16(s->x_qt)) || (s->w_qt && !aligned16(s->w_qt)))
        return set_error(FP8_ERR_ALIGN, "fp8_linear_fwd: tensors must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    const int f = recipe->fwd_format;

    if (recipe->scaling == FP8_SCALING_ROW) {
        // per-token X, per-output-channel W; with x_qt and w_qt kept (training)
        // the same launches also cast X^T and W^T per row (per column of X, W)
        if ((!s->x_sinv && M) || !s->w_sinv)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: per-row mode needs x_sinv and w_sinv");
        const bool keep = s->x_qt && s->w_qt;
        if (keep && (!s->x_sinv_t || !s->w_sinv_t))
            return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: per-row mode with x_qt/w_qt needs x_sinv_t and w_sinv_t");
        FP8_CHECK(cuda_status(launch_quantize_rows(X, M, K, f, recipe->pow2 != 0, s->x_q, s->x_sinv,
                                                   keep ? s->x_qt : nullptr, s->x_sinv_t, st),
                              "quantize X"));
        FP8_CHECK(cuda_status(launch_quantize_rows(W, N, K, f, recipe->pow2 != 0, s->w_q, s->w_sinv,
                                                   keep ? s->w_qt : nullptr, s->w_sinv_t, st),
                              "quantize W"));
        return launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_ROW, s->x_sinv, FP8_GRAN_ROW,
                           s->w_sinv, bias, Y, FP8_OUT_BF16, 0, st);
    }

    if (recipe->scaling == FP8_SCALING_BLOCK) {
        if ((!s->x_sinv && M) || !s->w_sinv)
            return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: block mode needs x_sinv and w_sinv");
        // training (x_qt and w_qt kept): the same casts also write the backward operands
        const bool keep = s->x_qt && s->w_qt;
        if (keep && (!s->x_sinv_t || !s->w_sinv_t))
            return set_error(FP8_ERR_INVALID_ARG, "fp8_linear_fwd: block mode with x_qt/w_qt needs x_sinv_t and w_sinv_t");
        if (keep && M % 128)
            return set_error(FP8_ERR_SHAPE, "fp8_linear_fwd: the block-wise backward operands need M multiple of 128");
        FP8_CHECK(cuda_status(launch_quantize_block(X, M, K, f, FP8_GRAN_1x128, recipe->pow2 != 0,
                                                    s->x_q, s->x_sinv, keep ? s->x_qt : nullptr,
                                                    s->x_sinv_t, st), "quantize X"));
        FP8_CHECK(cuda_status(launch_quantize_block(W, N, K, f, FP8_GRAN_128x128, recipe->pow2 != 0,
                                                    s->w_q, s->w_sinv, keep ? s->w_qt : nullptr,
                                                    s->w_sinv_t, st), "quantize W"));
        const int p2 = recipe->pow2 ? FP8_SCALE_POW2 : 0;
        return launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_1x128 | p2, s->x_sinv,
                           FP8_GRAN_128x128 | p2, s->w_sinv, bias, Y, FP8_OUT_BF16, 0, st);
    }

    FP8_CHECK(check_state_scales(s));
    const int H = history_len_of(recipe);
    if (recipe->scaling == FP8_SCALING_DYNAMIC) {
        if (!s->x_qt && !s->w_qt && M * K <= kSmallDynamicElems && N * K <= kSmallDynamicElems) {
            // a small layer: amax, scales and casts of X and W in one launch
            const ScaleUpd ux = dynamic_update(s, 0, recipe, s->qscale_inv + 0);
            const ScaleUpd uw = dynamic_update(s, 1, recipe, s->qscale_inv + 1);
            FP8_CHECK(cuda_status(launch_small_dynamic_cast(X, M * K, s->x_q, s->amax + 0, ux, W,
                                                            N * K, s->w_q, s->amax + 1, &uw, f, st),
                                  "amax and quantize X, W"));
            return launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_TENSOR, s->scale_inv + 0,
                               FP8_GRAN_TENSOR, s->scale_inv + 1, bias, Y, FP8_OUT_BF16, 0, st);
        }
        FP8_CHECK(cuda_status(launch_amax_pair(X, M * K, s->amax + 0, W, N * K, s->amax + 1, st),
                              "amax X, W"));
        if (!s->x_qt && !s->w_qt) {
            // one chunked cast of X and W that derives each scale from its amax
            // and writes the roles' updates itself ("scale computation" fused)
            const ScaleUpd ux = dynamic_update(s, 0, recipe, s->qscale_inv + 0);
            const ScaleUpd uw = dynamic_update(s, 1, recipe, s->qscale_inv + 1);
            FP8_CHECK(cuda_status(launch_quantize_pair(X, M, K, s->scale + 0, s->x_q, nullptr, nullptr,
                                                       W, N, K, s->scale + 1, s->w_q, nullptr, nullptr,
                                                       f, st, &ux, &uw),
                                  "quantize X, W"));
            return launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_TENSOR, s->scale_inv + 0,
                               FP8_GRAN_TENSOR, s->scale_inv + 1, bias, Y, FP8_OUT_BF16, 0, st);
        }
        FP8_CHECK(cuda_status(launch_update_scale(s->amax, s->history, s->pos, H, FP8_AMAX_MOST_RECENT,
                                                  f, recipe->margin, recipe->pow2 != 0, s->scale,
                                                  s->scale_inv, 2, st, s->qscale_inv, 1),
                              "update scales"));
        FP8_CHECK(cuda_status(quantize_x_w(X, W, M, N, K, f, s, false, st), "quantize X, W"));
        return launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_TENSOR, s->scale_inv + 0,
                           FP8_GRAN_TENSOR, s->scale_inv + 1, bias, Y, FP8_OUT_BF16, 0, st);
    }

    // delayed: cast with the scales of earlier steps, fold this step's amax in afterwards
    FP8_CHECK(cuda_status(quantize_x_w(X, W, M, N, K, f, s, true, st), "quantize X, W"));
    FP8_CHECK(launch_gemm(s->x_q, f, s->w_q, f, M, N, K, FP8_GRAN_TENSOR, s->scale_inv + 0,
                          FP8_GRAN_TENSOR, s->scale_inv + 1, bias, Y, FP8_OUT_BF16, 0, st));
    return cuda_status(launch_update_scale(s->amax, s->history, s->pos, H, recipe->amax_algo, f,
                                           recipe->margin, recipe->pow2 != 0, s->scale,
                                           s->scale_inv, 2, st, s->qscale_inv, 0),
                       "update scales");
}

int fp8_linear_bwd(const void* dY, int64_t M, int64_t N, int64_t K, const fp8_recipe_t* recipe,
                   const fp8_linear_state_t* s, void* dX, float* dW, int accumulate_dW,
                   float* dbias, void* workspace, size_t workspace_bytes, void* stream) {
    FP8_CHECK(check_linear_bwd_args(dY, M, N, K, recipe, s, dX, dW, dbias));
    FP8_CHECK(check_bwd_workspace(M, N, recipe, s, dbias, workspace, workspace_bytes));
    if (recipe->scaling == FP8_SCALING_BLOCK)
        return linear_bwd_block(dY, M, N, K, recipe, s, dX, dW, accumulate_dW, dbias, workspace,
                                as_stream(stream));
    if (recipe->scaling == FP8_SCALING_ROW)
        return linear_bwd_row(dY, M, N, K, recipe, s, dX, dW, accumulate_dW, dbias, workspace,
                              as_stream(stream));
    cudaStream_t st = as_stream(stream);
    // bias gradient: partial column sums fused into the (round-to-nearest) dY
    // cast, then summed in order; the stochastic cast leaves them to a pass
    // of their own
    float* partial = dbias ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                      bwd_operand_bytes(M, N, recipe, s))
                           : nullptr;
    float* fused_partial = recipe->sr_grad ? nullptr : partial;
    const int fb = recipe->bwd_format, ff = recipe->fwd_format;
    const int H = history_len_of(recipe);
    // With the forward's transposed copies (x_qt and w_qt both kept) the
    // backward GEMMs read K-major operands, dY_q^T included.  Without them
    // they read the codes as stored, MN-major: W_q [N x K] as dgrad's B,
    // dY_q [M x N] and X_q [M x K] as wgrad's A and B.
    const bool kmajor = s->x_qt && s->w_qt;
    uint8_t* dy_q = static_cast<uint8_t*>(workspace);
    uint8_t* dy_qt =
        kmajor ? dy_q + align256(static_cast<size_t>(M) * static_cast<size_t>(N)) : nullptr;
    float* h2 = s->history + 2 * static_cast<int64_t>(H);

    // dynamic scaling with the chunked cast (no transposed copy, no bias
    // sums, round to nearest): the cast derives the dY scale from its amax
    // and writes the role's update itself
    const bool fused_upd = recipe->scaling == FP8_SCALING_DYNAMIC && !recipe->sr_grad && !kmajor &&
                           !fused_partial;
    const bool small = fused_upd && M * N <= kSmallDynamicElems;
    if (recipe->scaling == FP8_SCALING_DYNAMIC && !small) {
        FP8_CHECK(cuda_status(launch_amax(dY, M * N, s->amax + 2, st), "amax dY"));
        if (!fused_upd)
            FP8_CHECK(cuda_status(launch_update_scale(s->amax + 2, h2, s->pos + 2, H,
                                                      FP8_AMAX_MOST_RECENT, fb, recipe->margin,
                                                      recipe->pow2 != 0, s->scale + 2,
                                                      s->scale_inv + 2, 1, st), "update dY scale"));
    }
    float* dy_amax = recipe->scaling == FP8_SCALING_DYNAMIC ? nullptr : s->amax + 2;
    if (recipe->sr_grad)   // "Stochastic rounding": unbiased gradient codes
        FP8_CHECK(cuda_status(launch_quantize_sr(dY, M, N, fb, s->scale + 2, 0, 0, dy_q, dy_qt,
                                                 dy_amax, st, s->sr_key), "quantize dY"));
    else if (small) {   // a small layer: amax, scale and cast of dY in one launch
        const ScaleUpd u = dynamic_update(s, 2, recipe, nullptr);
        FP8_CHECK(cuda_status(launch_small_dynamic_cast(dY, M * N, dy_q, s->amax + 2, u, nullptr,
                                                        0, nullptr, nullptr, nullptr, fb, st),
                              "amax and quantize dY"));
    } else if (fused_upd) {
        const ScaleUpd u = dynamic_update(s, 2, recipe, nullptr);
        FP8_CHECK(cuda_status(launch_quantize_pair(dY, M, N, s->scale + 2, dy_q, nullptr, nullptr,
                                                   nullptr, 0, 0, nullptr, nullptr, nullptr,
                                                   nullptr, fb, st, &u, nullptr),
                              "quantize dY"));
    } else
        FP8_CHECK(cuda_status(launch_quantize_tensor(dY, M, N, fb, s->scale + 2, dy_q, dy_qt,
                                                     dy_amax, st, nullptr, fused_partial),
                              "quantize dY"));
    if (dbias)
        FP8_CHECK(cuda_status(launch_dbias(dY, M, N, partial, fused_partial != nullptr, dbias,
                                           accumulate_dW, st), "dbias"));
    // dgrad: dX [M x K] = dY_q [M x N] . (W_q^T [K x N])^T, and
    // wgrad: dW [N x K] (+)= dY_q^T [N x M] . (X_q^T [K x M])^T, in one launch
    FP8_CHECK(launch_gemm_group(
        GemmArgs{dy_q, fb, kmajor ? s->w_qt : s->w_q, ff, M, K, N, FP8_GRAN_TENSOR,
                 s->scale_inv + 2, FP8_GRAN_TENSOR, s->qscale_inv + 1, nullptr, dX, FP8_OUT_BF16,
                 0, kmajor ? FP8_LAYOUT_TN : FP8_LAYOUT_B_KN},
        GemmArgs{kmajor ? dy_qt : dy_q, fb, kmajor ? s->x_qt : s->x_q, ff, N, K, M,
                 FP8_GRAN_TENSOR, s->scale_inv + 2, FP8_GRAN_TENSOR, s->qscale_inv + 0, nullptr,
                 dW, FP8_OUT_F32, accumulate_dW != 0, kmajor ? FP8_LAYOUT_TN : FP8_LAYOUT_KM_KN},
        st));
    if (recipe->scaling == FP8_SCALING_DELAYED)
        return cuda_status(launch_update_scale(s->amax + 2, h2, s->pos + 2, H, recipe->amax_algo, fb,
                                               recipe->margin, recipe->pow2 != 0, s->scale + 2,
                                               s->scale_inv + 2, 1, st), "update dY scale");
    return FP8_OK;
}

// Test hook, not part of the ABI that include/fp8linear.h declares: the
// time limit of the single-CTA GEMM kernel's epilogue wait for a full
// accumulator, in nanoseconds (default and maximum 2 s).  A test sets a short
// limit so that this bounded wait runs out on a long GEMM -- the kernel then
// returns early with bit 0 of fp8_device_status() set and the output left
// incomplete -- and restores the default afterwards.  The limit applies to
// kernels launched after the call on the current device.
int fp8_test_set_epilogue_wait_ns(uint64_t ns) {
    if (ns > 2000000000ull)
        return set_error(FP8_ERR_INVALID_ARG,
                         "fp8_test_set_epilogue_wait_ns: %llu ns is above the 2 s default",
                         static_cast<unsigned long long>(ns));
    return set_epilogue_wait_ns(ns);
}

int fp8_device_status(int* status, int clear) {
    if (!status) return set_error(FP8_ERR_INVALID_ARG, "fp8_device_status: NULL pointer");
    unsigned v = 0;
    FP8_CHECK(read_device_status(&v, clear != 0));
    *status = static_cast<int>(v);
    return FP8_OK;
}

}  // extern "C"
