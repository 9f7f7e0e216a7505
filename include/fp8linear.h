/*
 * fp8linear.h -- C ABI of the scaled FP8 linear layer for NVIDIA GB300 (sm_103a).
 *
 * The operation is the FP8 linear layer of mixed-precision LLM training as
 * "Mixed Precision LLM Training: The Complete Guide" describes it:
 *   forward   Y  = X . W^T            X [M x K], W [N x K] cast to E4M3
 *   dgrad     dX = dY . W             dY [M x N] cast to E5M2
 *   wgrad     dW (+)= dY^T . X        FP32 result, accumulated across calls
 * with FP32 accumulation inside every GEMM ("Skipping the BAcc accumulator
 * promotion"; "DeepSeek FP8 training recipe" > "Mixed-precision
 * accumulation"), per-tensor scales ("Transformer Engine internals" >
 * "Per-tensor scaling"), either current (dynamic) or delayed from an amax
 * history ("Delayed scaling", "History-based scaling"), or block-wise scales
 * ("DeepSeek FP8 training recipe" > "Block-wise scaling at 128
 * granularity").  Power-of-two scales follow the per-tensor "scaling bias"
 * of "Training and inference of large language models using 8-bit floating
 * point".
 *
 * Conventions shared by every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller.  Matrices are
 *     row-major and densely packed; bf16 tensors are passed as void*.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = the
 *     legacy default stream) and does no host synchronisation.  Scales,
 *     amaxes and histories stay in device memory; a call that reads a scale
 *     sees the value left by earlier work on the same stream.
 *   - The library allocates no device memory.  Calls that need scratch take
 *     a caller-owned `workspace` of at least fp8_workspace_size() bytes.
 *   - Return value: FP8_OK, or a negative status; on failure nothing was
 *     launched, except for FP8_ERR_CUDA, and fp8_last_error() returns a
 *     message (thread-local).
 *   - A tensor with no elements may be passed as NULL.
 *   - FP8 codes are round-to-nearest-even with saturation to the largest
 *     finite value (448 for E4M3, 57344 for E5M2); NaN becomes the code 0x7F.
 */
#ifndef FP8LINEAR_H
#define FP8LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- status */
#define FP8_OK               0
#define FP8_ERR_INVALID_ARG (-1)  /* null pointer, unknown enum, value out of range */
#define FP8_ERR_SHAPE       (-2)  /* a dimension violates the call's multiple-of rule */
#define FP8_ERR_ALIGN       (-3)  /* a pointer is not 16-byte aligned */
#define FP8_ERR_CUDA        (-4)  /* a CUDA call failed; see fp8_last_error() */
#define FP8_ERR_TIMEOUT     (-5)  /* a kernel's bounded wait gave up (device status) */
#define FP8_ERR_UNSUPPORTED (-6)  /* valid combination this library does not implement */

/* ------------------------------------------------------------------ enums */
typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format_t;
typedef enum { FP8_OUT_BF16 = 0, FP8_OUT_F32 = 1 } fp8_out_t;
typedef enum { FP8_AMAX_MAX = 0, FP8_AMAX_MOST_RECENT = 1 } fp8_amax_algo_t;
typedef enum {
    FP8_GRAN_TENSOR = 0,     /* one scale for the tensor                    */
    FP8_GRAN_1x128 = 1,      /* one scale per 128 consecutive row elements  */
    FP8_GRAN_128x128 = 2,    /* one scale per 128 x 128 tile                */
    FP8_GRAN_ROW = 3         /* one scale per row (per channel / token)     */
} fp8_gran_t;
/* Flag for fp8_gemm's ga / gb (and fp8_gemm_args_t), OR'd into
 * FP8_GRAN_1x128 or FP8_GRAN_128x128: every factor of that operand is a
 * power of two, as a cast with pow2 writes them (the per-tensor "scaling
 * bias" of "Training and inference of large language models using 8-bit
 * floating point", applied per block).  When both operands
 * carry it, the GEMM applies the factors inside the tensor core as UE8M0
 * block scales, each 128-deep block's factor on its four 32-deep steps: the
 * same terms, with one FP32 accumulation over all of K instead of a
 * promotion per 128-deep block.  Only the exponent of such a factor is read
 * (2^-127 and below read as 2^-127).  With one operand flagged, or with
 * other granularities, the flag changes nothing (it is rejected on
 * FP8_GRAN_TENSOR and FP8_GRAN_ROW). */
#define FP8_SCALE_POW2 16
/* Operand layouts of fp8_gemm.  The product is the same, D = A . B^T in the
 * [M x K] / [N x K] view; a layout only says how an operand is stored.  The
 * tensor core reads either form ("K-major" or "MN-major" tiles), so the
 * backward GEMMs can read the forward's codes as they are instead of
 * transposed copies. */
typedef enum {
    FP8_LAYOUT_TN = 0,       /* A [M x K] and B [N x K], both K-contiguous   */
    FP8_LAYOUT_B_KN = 1,     /* A [M x K]; B stored [K x N], N-contiguous    */
    FP8_LAYOUT_A_KM = 2,     /* A stored [K x M], M-contiguous; B [N x K]    */
    FP8_LAYOUT_KM_KN = 3     /* A stored [K x M] and B stored [K x N]        */
} fp8_layout_t;
typedef enum {
    FP8_SCALING_DELAYED = 0, /* per-tensor, scale from the amax history      */
    FP8_SCALING_DYNAMIC = 1, /* per-tensor, scale from the tensor's own amax */
    FP8_SCALING_BLOCK = 2,   /* 1x128 activations, 128x128 weights           */
    FP8_SCALING_ROW = 3      /* per-token X, per-output-channel W, per-token */
                             /* dY (dynamic), re-cast per column for bwd     */
} fp8_scaling_t;

/* Recipe of one linear layer ("Calibration deep dive" > "Dynamic
 * calibration": margin, amax_history_len, amax_compute_algo; "The HYBRID
 * recipe": E4M3 forward, E5M2 backward). */
typedef struct {
    int32_t scaling;      /* fp8_scaling_t                                   */
    int32_t margin;       /* 0..64: scale = fp8_max / amax / 2^margin        */
    int32_t history_len;  /* 1..1024, delayed scaling only                   */
    int32_t amax_algo;    /* fp8_amax_algo_t, delayed scaling only           */
    int32_t pow2;         /* nonzero: round scales down to powers of two     */
    int32_t fwd_format;   /* format of X and W (FP8_E4M3 for HYBRID)         */
    int32_t bwd_format;   /* format of dY (FP8_E5M2 for HYBRID)              */
    int32_t sr_grad;      /* 0 or 1: cast dY with stochastic rounding (the   */
                          /*   fp8_quantize_sr rule; per-tensor modes only,  */
                          /*   needs state->sr_key)                          */
} fp8_recipe_t;

/* Caller-owned device state of one linear layer.  Role r indexes the
 * per-tensor arrays: 0 = X (forward activation), 1 = W (forward weight),
 * 2 = dY (backward gradient) -- one scale per (tensor, format) pair
 * ("Transformer Engine internals" > "Per-tensor scaling").  Everything here
 * is plain device memory, so checkpointing the layer means copying it. */
typedef struct {
    float*   scale;      /* [3] quantisation scales, initialise to 1           */
    float*   scale_inv;  /* [3] 1/scale, initialise to 1                       */
    float*   amax;       /* [3] out: max|x| of the last tensor of each role    */
    float*   history;    /* [3][H] amax history (H = history_len, 1 for        */
                         /*   dynamic), initialise to 0                        */
    int32_t* pos;        /* [3] next history slot, initialise to 0             */
    uint8_t* x_q;        /* [M][K] written by fwd                              */
    uint8_t* x_qt;       /* [K][M] written by fwd; nullable in per-tensor      */
                         /*   modes (see fp8_linear_bwd)                       */
    uint8_t* w_q;        /* [N][K] written by fwd                              */
    uint8_t* w_qt;       /* [K][N] written by fwd; nullable in per-tensor modes*/
    float*   x_sinv;     /* [M][K/128] written by fwd (block mode)             */
    float*   w_sinv;     /* [N/128][K/128] written by fwd (block mode)         */
    float*   qscale_inv; /* [2] out: dequantisation factors that x_q/x_qt (0)  */
                         /*   and w_q/w_qt (1) were cast with; written by fwd  */
                         /*   (per-tensor modes), read by bwd                  */
    float*   x_sinv_t;   /* [K][M/128] block mode: scales of x_qt, the 1x128   */
                         /*   block cast of X^T (blocks run along the tokens)  */
    float*   w_sinv_t;   /* [K/128][N/128] block mode: scales of w_qt = W_q^T  */
    uint64_t* sr_key;    /* [2] with recipe->sr_grad: (seed, counter) of the   */
                         /*   stochastic dY cast, i.e. fp8_quantize_sr's seed  */
                         /*   and offset; each backward call uses the counter  */
                         /*   and then adds 1 to it on the device              */
} fp8_linear_state_t;

/* ---------------------------------------------------------------- calls */

/* amax = max |x| over n bf16 values ("Per-tensor scaling": the scale is set
 * from the tensor's max absolute value).  Computed as an integer max over
 * the |bf16| bit patterns: exact and independent of order; any NaN gives
 * NaN.  x: 16-byte aligned, n >= 0 (n = 0 gives 0).  amax: one float,
 * overwritten. */
int fp8_amax(const void* x, int64_t n, float* amax, void* stream);

/* One step of the scale update ("Delayed scaling", "History-based scaling";
 * "torch.compile and FP8" for the all-zero skip):
 *   history[*pos] = *amax;  *pos = (*pos + 1) % history_len;
 *   a = (algo == FP8_AMAX_MAX) ? max(history) : *amax;
 *   if a is 0 or not finite: *scale and *scale_inv are left unchanged;
 *   else  s = fp8_max(format) / a            (fp32, round to nearest)
 *         s = s * 2^-margin                  (fp32)
 *         s = min(max(s, FLT_MIN), FLT_MAX)
 *         if pow2: s = 2^floor(log2 s)
 *         *scale = s;  *scale_inv = 1 / s    (fp32, round to nearest).
 * amax values are magnitudes (>= 0 or NaN).  history_len 1..1024, margin
 * 0..64.  Dynamic scaling is history_len = 1.  All pointers device. */
int fp8_update_scale(const float* amax, float* history, int32_t* pos, int history_len,
                     int algo, int format, int margin, int pow2, float* scale,
                     float* scale_inv, void* stream);

/* Cast a bf16 matrix x [rows x cols] to FP8.
 * granularity FP8_GRAN_TENSOR: q = fp8(fp32(x) * (*scale)), one fp32 multiply
 *   then the saturating round-to-nearest-even cast ("Per-tensor scaling").
 *   q_t (nullable) receives the transpose [cols x rows] in the same launch;
 *   amax_out (nullable) receives max|x| (fused reduction, overwritten).
 *   Shape rule: rows*cols any when q_t is NULL; with q_t, rows and cols must
 *   be multiples of 16.
 * granularity FP8_GRAN_1x128 / FP8_GRAN_128x128: each 1x128 row segment or
 *   128x128 tile gets its own scale fp8_max/amax_block (margin 0; 1 for an
 *   all-zero or non-finite block; rounded down to a power of two if pow2),
 *   and scale_inv_blocks receives 1/scale as [rows/b][cols/128] (b = 1 or
 *   128) ("Block-wise scaling at 128 granularity").  scale and amax_out must
 *   be NULL.  cols must be a multiple of 128 (and rows, for 128x128).
 *   q_t (nullable; rows a multiple of 128; with scale_inv_blocks_t) gets, in
 *   the same pass,
 *     1x128:   the 1x128 block cast of x^T [cols x rows] -- blocks of 128
 *              consecutive rows of one column of x -- with scale_inv_blocks_t
 *              [cols][rows/128] (the operand layout of the wgrad GEMM);
 *     128x128: the transposed codes (a 128x128 block keeps its scale) with
 *              the transposed scales scale_inv_blocks_t [cols/128][rows/128].
 * granularity FP8_GRAN_ROW ("Transformer Engine internals" > "Per-row vs
 *   per-tensor scaling"): one scale per row, fp8_max / amax_row by the block
 *   rule; scale_inv_blocks [rows].  q_t (with scale_inv_blocks_t, rows a
 *   multiple of 16) gets the per-row cast of x^T -- one scale per column of x
 *   -- with scale_inv_blocks_t [cols].  cols must be a multiple of 16.
 * x, q, q_t: 16-byte aligned.  format: FP8_E4M3 or FP8_E5M2. */
int fp8_quantize(const void* x, int64_t rows, int64_t cols, int format, int granularity,
                 const float* scale, int pow2, uint8_t* q, uint8_t* q_t,
                 float* scale_inv_blocks, float* scale_inv_blocks_t, float* amax_out,
                 void* stream);

/* Per-tensor cast (FP8_GRAN_TENSOR semantics of fp8_quantize, same q, q_t
 * and amax_out) with the dashboard counters of "Numerical-failure taxonomy"
 * > "A diagnostic dashboard" fused into the same pass:
 *   counts[0] += inputs x != +-0 whose FP8 code is +-0 (flushed to zero:
 *                the numerator of the underflow ratio)
 *   counts[1] += inputs whose scaled value |fp32(x) * scale| exceeds the
 *                largest finite FP8 value (saturated; +-Inf included, NaN not)
 * counts: 2 x uint64 in device memory, accumulated (zero it to start a count). */
int fp8_quantize_counted(const void* x, int64_t rows, int64_t cols, int format,
                         const float* scale, uint8_t* q, uint8_t* q_t, float* amax_out,
                         unsigned long long* counts, void* stream);

/* Per-tensor cast (FP8_GRAN_TENSOR semantics of fp8_quantize: same scale,
 * q, q_t, amax_out and shape rules) with stochastic rounding instead of
 * round-to-nearest-even ("Mixed Precision LLM Training: The Complete
 * Guide", "Stochastic rounding": round up or down at random, with the
 * probability given by the remainder, so the cast is unbiased).
 *   v = fp32(x) * scale (one fp32 multiply), lo <= |v| <= hi its two FP8
 *   neighbours, f = (|v| - lo) / (hi - lo); the magnitude becomes hi iff
 *   r < floor(f * 2^32), r a uniform 32-bit word, so P(hi) = f exactly
 *   in the normal FP8 range.  Saturating to the largest finite value; NaN ->
 *   0x7F; zeros keep their sign.
 *   r for element i (row-major index i = row * cols + col) is word (i mod 4)
 *   of Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 *   as easy as 1, 2, 3", SC'11) at counter (lo32(i/4), hi32(i/4),
 *   lo32(offset), hi32(offset)) and key (lo32(seed), hi32(seed)).  The codes
 *   depend only on (x, scale, seed, offset), not on the launch; q_t holds the
 *   same codes as q, transposed.  Advance offset (or change seed) between
 *   casts that need independent draws.
 * Errors as fp8_quantize. */
int fp8_quantize_sr(const void* x, int64_t rows, int64_t cols, int format, const float* scale,
                    uint64_t seed, uint64_t offset, uint8_t* q, uint8_t* q_t, float* amax_out,
                    void* stream);

/* Scaled FP8 GEMM:
 *   D[m][n] = sum_k sa(m,k) * sb(n,k) * A[m][k] * B[n][k]
 * where A[m][k] is the byte at A + m*K + k (FP8_LAYOUT_TN, FP8_LAYOUT_B_KN)
 * or at A + k*M + m (FP8_LAYOUT_A_KM, FP8_LAYOUT_KM_KN), and B[n][k] the
 * byte at B + n*K + k or, with FP8_LAYOUT_B_KN / FP8_LAYOUT_KM_KN, at
 * B + k*N + n.  The layouts other than FP8_LAYOUT_TN take per-tensor and
 * per-row factors (FP8_ERR_UNSUPPORTED with block factors).
 * with FP32 accumulation on the tensor cores.  sa, sb are DEQUANTISATION
 * factors (scale_inv = 1/scale, device memory):
 *   FP8_GRAN_TENSOR   scale_inv[0]
 *   FP8_GRAN_1x128    scale_inv[row][k/128]
 *   FP8_GRAN_128x128  scale_inv[row/128][k/128]
 *   FP8_GRAN_ROW      scale_inv[row]
 * (a row of B is a column n of D: 1x128 or per-row scales on B scale D
 * column-wise).  Per-row factors are applied like per-tensor ones, in the
 * epilogue: D[m][n] = fp32(sa[m] * sb[n]) * acc[m][n]; they cannot be mixed
 * with block scales (FP8_ERR_UNSUPPORTED).
 * Per-tensor factors multiply the FP32 result once; block factors scale each
 * 128-deep partial sum before it is added ("applied during the matmul").
 * bias (nullable): bf16 [N], 16-byte aligned, added in FP32 to every row of
 * the scaled result before the output rounding (te.Linear's bias, "Mixed
 * Precision LLM Training: The Complete Guide", "Transformer Engine
 * internals"): D[m][n] = fp32(factors * acc[m][n]) + bias[n].
 * out FP8_OUT_BF16: D is bf16 [M x N], rounded to nearest even.
 * out FP8_OUT_F32:  D is fp32 [M x N]; accumulate != 0 adds to D.
 * Shape rule: M >= 0; N, K multiples of 16 (multiples of 128 when either
 * operand uses block scales); M a multiple of 16 when A is stored [K x M].
 * A, B, D: 16-byte aligned.  An unknown layout is FP8_ERR_INVALID_ARG.
 * fa, fb: FP8_E4M3 / FP8_E5M2 in any combination. */
int fp8_gemm(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
             int64_t K, int layout, int ga, const float* scale_inv_a, int gb,
             const float* scale_inv_b, const void* bias, void* D, int out, int accumulate,
             void* stream);

/* The arguments of one fp8_gemm call, for fp8_gemm_group. */
typedef struct {
    const uint8_t* A;
    int32_t fa;
    const uint8_t* B;
    int32_t fb;
    int64_t M, N, K;
    int32_t layout;
    int32_t ga;
    const float* scale_inv_a;
    int32_t gb;
    const float* scale_inv_b;
    const void* bias;
    void* D;
    int32_t out;
    int32_t accumulate;
} fp8_gemm_args_t;

/* Two independent GEMMs in one launch: the same results, bit for bit, as
 * fp8_gemm(g1) followed by fp8_gemm(g2).  When both are per-tensor / per-row
 * problems without bias whose 128 x 128 tiles fit together in one wave (at
 * most one per SM), one single-CTA launch takes both problems' tiles; when
 * both have at least 256 rows or an MN-major operand, one persistent CTA-pair
 * grid deals both problems' 256 x 256 tiles from one list, the deeper
 * problem's first, so that neither leaves a partly filled last wave of its
 * own (the dgrad and wgrad of a backward pass are such a pair); otherwise
 * the two run as two launches.  The problems run concurrently: neither may read or
 * write the other's output.  Each is validated as by fp8_gemm; NULL g1 or
 * g2 is FP8_ERR_INVALID_ARG.  (The pages have no counterpart: this is a
 * scheduling property of the library -- the dgrad and wgrad GEMMs of
 * "Transformer Engine internals" computed together -- not of the method.) */
int fp8_gemm_group(const fp8_gemm_args_t* g1, const fp8_gemm_args_t* g2, void* stream);

/* Bytes of workspace that fp8_linear_bwd needs for a layer of this shape
 * and recipe: the quantised dY operands (and their scale arrays), plus
 * 4*ceil(M/128)*N bytes for the bias gradient's partial sums, which only a
 * call with dbias uses.  fp8_linear_fwd needs none.  Returns 0 for an
 * invalid recipe.  This is the size for either per-tensor backward; one
 * whose state keeps no transposed copies needs M*N code bytes fewer (a
 * smaller workspace is accepted then). */
size_t fp8_workspace_size(int64_t M, int64_t N, int64_t K, const fp8_recipe_t* recipe);

/* Forward pass Y [M x N] (bf16) = X [M x K] . W [N x K]^T (+ bias [N], bf16,
 * nullable, 16-byte aligned, added in the GEMM epilogue in FP32).
 *   delayed: quantise X and W with the current scales (fusing their amax,
 *            and their transposes when x_qt / w_qt are set), GEMM, then
 *            update the X and W scales (the new scales take effect on the
 *            next call: one-step lag);
 *   dynamic: amax, scale update and quantisation of X and W, then GEMM;
 *   row:     per-token scales for X and per-output-channel scales for W (the
 *            state's x_sinv [M], w_sinv [N]), GEMM with vector factors; with
 *            x_qt and w_qt set, also the per-row casts of X^T and W^T (one
 *            scale per column of X and W: x_sinv_t [K], w_sinv_t [K]), which
 *            the backward's reductions need;
 *   block:   1x128 quantisation of X, 128x128 of W, block-scaled GEMM; with
 *            state->x_qt and w_qt set (training) the same passes also write
 *            the 1x128 block cast of X^T (x_qt, x_sinv_t) and W_q^T (w_qt,
 *            w_sinv_t) for the backward pass, which needs M % 128 == 0.
 * Writes state->x_q/x_qt/w_q/w_qt (and the block scale arrays) for the
 * backward pass.  Shape rule: M, N, K multiples of 16 (N, K multiples of 128
 * for block).  M = 0 (a batch without tokens, e.g. an expert that received
 * none) is a valid call: X, Y and the state's M-sized arrays (x_q, x_qt,
 * x_sinv) may then be NULL; W is cast and the scaling state advances as for
 * any batch, with an amax of 0 for X (so its scale update is skipped). */
int fp8_linear_fwd(const void* X, const void* W, const void* bias, int64_t M, int64_t N,
                   int64_t K, const fp8_recipe_t* recipe, const fp8_linear_state_t* state,
                   void* Y, void* workspace, size_t workspace_bytes, void* stream);

/* Backward pass after fp8_linear_fwd on the same state:
 *   dX [M x K] (bf16) = dY . W,   dW [N x K] (fp32) = dY^T . X  (+ dW if
 *   accumulate_dW).  dY is cast to the recipe's bwd_format with the dY
 *   role's scale (delayed: current scale, then update; dynamic: its own
 *   amax).  The quantised dY (and its transpose) live in the workspace.
 * Per-tensor scaling: with both x_qt and w_qt set the backward GEMMs read
 *   the transposed copies (K-major operands, dY_q^T included, as in
 *   "Transformer Engine internals"); with either one NULL they read x_q,
 *   w_q and dY_q as stored (FP8_LAYOUT_B_KN for dgrad, FP8_LAYOUT_KM_KN for
 *   wgrad) and no transposed copy is made.  Both give the same codes and
 *   the same GEMM results.
 * M = 0 (no tokens): dY and dX may be NULL (so may the forward's M-sized
 *   arrays); dY's amax is 0 (its scale update is skipped), dW and dbias are
 *   set to zero, or left as they are with accumulate_dW, and the workspace
 *   may be NULL when fp8_workspace_size gives 0.
 * Block scaling ("DeepSeek FP8 training recipe" > "Block-wise scaling at
 *   128 granularity"): dY is cast once into 1x128 blocks along N (dgrad
 *   operand) and 1x128 blocks along the tokens of dY^T (wgrad operand);
 *   dgrad = block GEMM with W_q^T's 128x128 scales; wgrad = block GEMM of
 *   dY^T and X^T, both with 1x128 scales along the tokens.  Needs the
 *   forward pass to have kept x_qt/x_sinv_t and w_qt/w_sinv_t, and
 *   M % 128 == 0.  Workspace: 2*M*N code bytes + 8*M*N/128 scale bytes.
 * Per-row scaling: dY is cast per token (dgrad, with W^T's per-input-channel
 *   cast) and per output channel (dY^T, wgrad, with X^T's per-input-channel
 *   cast); workspace 2*M*N code bytes + 4*(M+N) scale bytes.
 * dbias (nullable, fp32 [N], 4-byte aligned): the bias gradient, the column
 *   sums of dY, dbias[n] = sum_m dY[m][n] (+ dbias[n] if accumulate_dW),
 *   summed in FP32 in a fixed order (per 128-token tile, then over the
 *   tiles), so repeated calls give identical bits.  With per-tensor scaling
 *   the tile sums come out of the dY cast's own pass; the block-wise and
 *   per-row modes read dY once more.  Needs the partial-sum part of
 *   fp8_workspace_size(). */
int fp8_linear_bwd(const void* dY, int64_t M, int64_t N, int64_t K,
                   const fp8_recipe_t* recipe, const fp8_linear_state_t* state, void* dX,
                   float* dW, int accumulate_dW, float* dbias, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Size of the built-in device scratch of fp8_linear_bwd_noalloc: 32 MiB. */
#define FP8_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* fp8_linear_bwd for callers that cannot allocate device memory -- e.g. an
 * operator inside a host framework whose memory planner owns every device
 * buffer and passes it only its inputs and outputs, a latency-critical caller
 * that must avoid cudaMalloc's implicit synchronisation, or a process whose
 * caching allocator has reserved almost all device memory.  (The pages have
 * no counterpart: this is a property of the library, not of the method.)
 * Same arguments and results as fp8_linear_bwd, minus the workspace and the
 * bias gradient (dbias = NULL): the
 * quantised gradient (and its transpose, where the backward makes one) goes
 * to a fixed device array of FP8_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Shapes whose dY operands exceed it are rejected with FP8_ERR_SHAPE and a
 * message naming the limit: with per-tensor scaling M*N > 32 MiB (e.g. more
 * than 4096 x 8192) without transposed copies, 2*M*N > 32 MiB with them.
 * Calls no allocating routine.  Arguments are checked first: a call that
 * fails them returns its status without touching the device.  The first
 * call in each CUDA context (normally the device's primary context: once
 * per device) looks up the array's device address (cudaGetSymbolAddress)
 * with that context current and keeps it under the context's unique ID, so
 * a context made after cudaDeviceReset, or one the caller makes current,
 * gets its own lookup; make that first call before any stream capture.
 * Every call on a device shares the array and leaves its contents behind;
 * calls whose work overlaps on the GPU race on it, so order them on one
 * stream. */
int fp8_linear_bwd_noalloc(const void* dY, int64_t M, int64_t N, int64_t K,
                           const fp8_recipe_t* recipe, const fp8_linear_state_t* state,
                           void* dX, float* dW, int accumulate_dW, void* stream);

/* Message of the last failing call on this host thread ("" if none). */
const char* fp8_last_error(void);

/* Read (and, if clear != 0, reset) the device status word that kernels set:
 *   bit 0 (1): a bounded wait gave up (timeout);
 *   bit 1 (2): a scale update met a non-finite amax -- a NaN or Inf in a
 *              cast tensor, or still in its amax history -- and kept the
 *              previous scale ("Numerical-failure taxonomy": NaN / Inf are
 *              caught at the first step that sees them).
 * Synchronises the device.  Returns FP8_OK and *status = 0 when every
 * kernel finished normally. */
int fp8_device_status(int* status, int clear);

#ifdef __cplusplus
}
#endif
#endif /* FP8LINEAR_H */
