// noalloc.cu -- fp8_linear_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// fp8_linear_bwd needs scratch for the quantised gradient (M x N bytes, and
// as much again for its transpose when the state keeps transposed copies or
// the recipe is block-wise or per-row), and asks the caller for it as a
// workspace.  Some callers
// have no way to provide one: a custom operator inside a host framework whose
// memory planner owns every device buffer and hands the operator only its
// inputs and outputs; a latency-critical caller that must not pay for
// cudaMalloc's implicit device synchronisation; a process whose caching
// allocator has already reserved nearly all device memory, so that a raw
// cudaMalloc fails although the pool has room.  For them the scratch lives in
// this file's own device array, sized once when the library is loaded.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Nothing in it has to start at zero: the gradient cast writes
// every byte of both layouts before the GEMMs read them.  Calls whose work
// overlaps on the GPU (e.g. issued on two streams without ordering) race on
// the array and must be serialised by the caller.
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fp8linear.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = FP8_NOALLOC_SCRATCH_BYTES;

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) uint8_t g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
std::vector<std::pair<unsigned long long, void*>> g_scratch_by_ctx;   // (context ID, address)

// Device address of g_bwd_scratch in the current context.  The host-side
// symbol is only a stand-in, and the module -- with the array -- is loaded
// once per context, so the address is looked up (cudaGetSymbolAddress, with
// the context current) on the first call in each context and kept under that
// context's ID.
int scratch_in_current_context(void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = fp8::current_context_id();
    if (id != 0) {
        for (const auto& e : g_scratch_by_ctx)
            if (e.first == id) {
                *out = e.second;
                return FP8_OK;
            }
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || !p)
        return fp8::set_error(FP8_ERR_CUDA, "fp8_linear_bwd_noalloc: cudaGetSymbolAddress: %s",
                              cudaGetErrorString(e));
    // the lookup made the device's primary context current if none was
    const unsigned long long id_now = id != 0 ? id : fp8::current_context_id();
    if (id_now != 0) g_scratch_by_ctx.emplace_back(id_now, p);
    *out = p;
    return FP8_OK;
}

}  // namespace

extern "C" int fp8_linear_bwd_noalloc(const void* dY, int64_t M, int64_t N, int64_t K,
                                      const fp8_recipe_t* recipe,
                                      const fp8_linear_state_t* state, void* dX, float* dW,
                                      int accumulate_dW, void* stream) {
    // every argument check first: a call that fails them touches no device
    // state (no context is made current, no module is loaded)
    const int bad = fp8::check_linear_bwd_args(dY, M, N, K, recipe, state, dX, dW, nullptr);
    if (bad != FP8_OK) return bad;
    // the dY operands only: this entry point computes no bias gradient
    const size_t need = fp8::bwd_operand_workspace(M, N, recipe, state);
    if (need > kScratchBytes)
        return fp8::set_error(FP8_ERR_SHAPE,
                              "fp8_linear_bwd_noalloc: M x N = %lld x %lld needs %zu bytes of "
                              "scratch; the built-in scratch holds %zu bytes",
                              static_cast<long long>(M), static_cast<long long>(N), need,
                              kScratchBytes);
    void* scratch = nullptr;
    const int st = scratch_in_current_context(&scratch);
    if (st != FP8_OK) return st;
    return fp8_linear_bwd(dY, M, N, K, recipe, state, dX, dW, accumulate_dW, nullptr, scratch,
                          kScratchBytes, stream);
}

// Test hook, not part of the ABI that include/fp8linear.h declares: the
// scratch address that fp8_linear_bwd_noalloc would use in the current
// context (*cached, from the per-context table) and a fresh lookup of the
// array's address in that context (*fresh).  The two must agree in every
// context, also after other contexts have been used.
extern "C" int fp8_test_noalloc_scratch(void** cached, void** fresh) {
    if (!cached || !fresh)
        return fp8::set_error(FP8_ERR_INVALID_ARG, "fp8_test_noalloc_scratch: NULL pointer");
    const int st = scratch_in_current_context(cached);
    if (st != FP8_OK) return st;
    const cudaError_t e = cudaGetSymbolAddress(fresh, g_bwd_scratch);
    if (e != cudaSuccess)
        return fp8::set_error(FP8_ERR_CUDA, "fp8_test_noalloc_scratch: cudaGetSymbolAddress: %s",
                              cudaGetErrorString(e));
    return FP8_OK;
}
