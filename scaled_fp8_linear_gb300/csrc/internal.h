// internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments are validated by the caller; these
// functions only configure and enqueue kernels on `stream`.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/fp8linear.h"

namespace fp8 {

// Launch `kernel` on `stream` with programmatic stream serialisation: it may
// start while the previous kernel of the stream finishes, and it waits for
// that kernel (griddepcontrol.wait) before touching global memory -- every
// kernel of this library does.  Errors are also left for cudaGetLastError().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor map of a row-major bf16 matrix [rows x cols] for TMA loads of
// box_rows x box_cols boxes (no swizzle; zero fill outside the matrix).
// FP8_OK or a status with its message.
int make_bf16_box_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols,
                      uint32_t box_cols, uint32_t box_rows);

// Number of SMs of the current device (cached per device).
int num_sms();

// max|x| over n bf16 values into *amax (zeroed first, then atomically raised).
cudaError_t launch_amax(const void* x, int64_t n, float* amax, cudaStream_t stream);

// The amaxes of two tensors (x1 may be empty, amax1 then nullable) in one
// zeroing launch and one amax launch.
cudaError_t launch_amax_pair(const void* x0, int64_t n0, float* amax0, const void* x1, int64_t n1,
                             float* amax1, cudaStream_t stream);

// Scale update for `nroles` consecutive roles of a state laid out as
// amax[r], history[r * H + i], pos[r], scale[r], scale_inv[r].  `saved`
// (nullable) receives scale_inv[r] from before (save_after = 0) or after
// (save_after = 1) the update.
cudaError_t launch_update_scale(const float* amax, float* history, int32_t* pos, int H,
                                int algo, int fmt, int margin, int pow2, float* scale,
                                float* scale_inv, int nroles, cudaStream_t stream,
                                float* saved = nullptr, int save_after = 0);

// Per-tensor cast of x [rows x cols]; q_t and amax may be null.  With q_t,
// rows and cols are multiples of 16.
// counts (nullable): the cast's dashboard counters [underflow, saturated] are
// added to counts[0..1].
// dbias_partial (nullable; needs q_t): the same pass also writes the bias
// gradient's partial column sums, one row of `cols` floats per 128-row tile.
cudaError_t launch_quantize_tensor(const void* x, int64_t rows, int64_t cols, int fmt,
                                   const float* scale, uint8_t* q, uint8_t* q_t, float* amax,
                                   cudaStream_t stream, unsigned long long* counts = nullptr,
                                   float* dbias_partial = nullptr);

// Dynamic scaling's update of one role, taken inside a cast kernel instead
// of a launch of its own: every CTA derives the scale from the role's amax
// (written by the amax pass before the cast) as the update kernel does
// (history length 1, most recent), and the first CTA writes the role's
// history, pos, scale and scale_inv (and `saved`, when set, after the
// update).  An amax that is 0 or not finite leaves the scale as it was (a
// non-finite one sets bit 1 of `status`).
struct ScaleUpd {
    const float* amax;   // null: no update, the cast reads *scale
    float* history;
    int32_t* pos;
    int margin;
    int pow2;
    float* scale;
    float* scale_inv;
    float* saved;
    unsigned* status;
};

// Dynamic scaling of up to two small tensors (n0, n1 <= kSmallDynamicElems
// elements; the second optional: upd1 null) in one launch: each tensor's
// amax (written to amax0 / amax1), its scale and state update per the
// ScaleUpd (whose amax field is not read), and its codes q0 / q1 -- the same
// bits as the amax pass followed by the chunked cast with a fused update.
constexpr int64_t kSmallDynamicElems = int64_t{1} << 20;
cudaError_t launch_small_dynamic_cast(const void* x0, int64_t n0, uint8_t* q0, float* amax0,
                                      const ScaleUpd& upd0, const void* x1, int64_t n1,
                                      uint8_t* q1, float* amax1, const ScaleUpd* upd1, int fmt,
                                      cudaStream_t stream);

// Per-tensor casts of two tensors in one launch (x0 and x1 each [rows x
// cols]), both to `fmt`: with transposes (qt0 and qt1 set; rows and cols
// multiples of 16), or without (both null: the chunked cast, any size).
// amax0 and amax1 both null or both set (zeroed first).  upd0 / upd1
// (chunked cast only, nullable): the dynamic update of each tensor's role,
// fused into the cast; scale0 / scale1 are then that role's scale.
cudaError_t launch_quantize_pair(const void* x0, int64_t rows0, int64_t cols0, const float* scale0,
                                 uint8_t* q0, uint8_t* qt0, float* amax0, const void* x1,
                                 int64_t rows1, int64_t cols1, const float* scale1, uint8_t* q1,
                                 uint8_t* qt1, float* amax1, int fmt, cudaStream_t stream,
                                 const ScaleUpd* upd0 = nullptr, const ScaleUpd* upd1 = nullptr);

// Bias gradient dbias[n] (+)= sum_m x[m][n] of a bf16 x [rows x cols]
// (cols % 16 == 0), in fp32 and a fixed order.  partial: ceil(rows/128) x
// cols floats of workspace, already filled by a fused cast when
// partial_ready, else filled here from x first.
cudaError_t launch_dbias(const void* x, int64_t rows, int64_t cols, float* partial,
                         bool partial_ready, float* dbias, int accumulate, cudaStream_t stream);

// Per-tensor cast of launch_quantize_tensor with stochastic rounding: element
// i (row-major) draws word i % 4 of Philox-4x32-10(counter = (i / 4, offset),
// key = seed).  key_dev (nullable): take (seed, offset) from key_dev[0..1]
// in device memory instead, and add 1 to key_dev[1] after the cast.
cudaError_t launch_quantize_sr(const void* x, int64_t rows, int64_t cols, int fmt,
                               const float* scale, uint64_t seed, uint64_t offset, uint8_t* q,
                               uint8_t* q_t, float* amax, cudaStream_t stream,
                               uint64_t* key_dev = nullptr);

// Block cast: gran 1 (1x128) or 2 (128x128); writes q and 1/scale per block.
// q_t (nullable, rows % 128 == 0): gran 1 -> the 1x128 block cast of x^T with
// scale_inv_t [cols][rows/128]; gran 2 -> the transposed codes with the
// transposed scales scale_inv_t [cols/128][rows/128].
cudaError_t launch_quantize_block(const void* x, int64_t rows, int64_t cols, int fmt, int gran,
                                  int pow2, uint8_t* q, float* scale_inv, uint8_t* q_t,
                                  float* scale_inv_t, cudaStream_t stream);

// Per-row cast: q with one scale per row (scale_inv [rows]); q_t (nullable,
// rows and cols multiples of 16) is the per-row cast of x^T, i.e. one scale
// per column of x (scale_inv_t [cols]).  cols is a multiple of 8.
cudaError_t launch_quantize_rows(const void* x, int64_t rows, int64_t cols, int fmt, int pow2,
                                 uint8_t* q, float* scale_inv, uint8_t* q_t, float* scale_inv_t,
                                 cudaStream_t stream);

// Scaled FP8 GEMM.  layout: FP8_LAYOUT_TN (A [M x K], B [N x K]), or with
// FP8_LAYOUT_A_KM / FP8_LAYOUT_B_KN an operand stored [K x M] / [K x N]
// (per-tensor and per-row scales only).  Returns 0 or a negative fp8 status
// code (tensor-map encoding can fail); launch errors come back as
// FP8_ERR_CUDA.  bias (nullable): bf16 [N] added to every row before the
// output rounding.
int launch_gemm(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                int64_t K, int ga, const float* sa, int gb, const float* sb, const void* bias,
                void* D, int out, int accumulate, cudaStream_t stream,
                int layout = FP8_LAYOUT_TN);

// Workspace bytes of fp8_linear_bwd's dY operands (without the bias
// gradient's partial sums) for a valid recipe; with a state (nullable), what
// that state's per-tensor backward needs (dY_q alone when it keeps no
// transposed copies).
size_t bwd_operand_workspace(int64_t M, int64_t N, const fp8_recipe_t* recipe,
                             const fp8_linear_state_t* s = nullptr);

// Every check that fp8_linear_bwd makes before it looks at its workspace:
// recipe, shape, the state pointers the recipe's mode needs, alignment.
// FP8_OK or the status (with its message) that fp8_linear_bwd would return.
int check_linear_bwd_args(const void* dY, int64_t M, int64_t N, int64_t K,
                          const fp8_recipe_t* recipe, const fp8_linear_state_t* s, const void* dX,
                          const float* dW, const float* dbias);

// The arguments of one launch_gemm call.
struct GemmArgs {
    const uint8_t* A;
    int fa;
    const uint8_t* B;
    int fb;
    int64_t M, N, K;
    int ga;
    const float* sa;
    int gb;
    const float* sb;
    const void* bias;
    void* D;
    int out;
    int accumulate;
    int layout = FP8_LAYOUT_TN;
};

// Two independent GEMMs of one pass (the dgrad and the wgrad of a backward)
// in one persistent launch of the CTA-pair kernel: both problems' tiles are
// dealt to the clusters from one list, the deeper problem's first, so that
// neither leaves a partly filled last wave of its own.  Falls back to two
// launch_gemm calls when either problem is not a CTA-pair problem.
int launch_gemm_group(const GemmArgs& g1, const GemmArgs& g2, cudaStream_t stream);

// Device status word (bit 0: a bounded wait timed out; bit 1: a scale
// update saw a non-finite amax).
int read_device_status(unsigned* status, bool clear);

// Sets the epilogue wait limit of the single-CTA GEMM kernel on the current
// device (g_epilogue_wait_ns; synchronous).
int set_epilogue_wait_ns(uint64_t ns);

// Unique ID of the calling thread's current CUDA context (cuCtxGetId), 0 if
// there is none or it cannot be read.  IDs are never reused within a
// process, so caches of device addresses keyed by it stay valid across
// cudaDeviceReset and across contexts a caller makes current.
unsigned long long current_context_id();

// Device address of the status word in the current context (null if it
// cannot be looked up), for kernels outside gemm.cu to set bits in.
unsigned* device_status_word();

// Record a message for fp8_last_error() and return `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace fp8
