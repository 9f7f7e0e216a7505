// gemm.cu -- the compute-bound half of the scaled FP8 linear: FP8 x FP8 GEMMs
// on the sm_103a tensor cores (tcgen05.mma kind::f8f6f4), fed by TMA through
// a shared-memory ring, accumulating in TMEM (FP32), with the dequantisation
// fused into the epilogue.
//
// Method ("Mixed Precision LLM Training: The Complete Guide"):
//   "Transformer Engine internals" > "Per-tensor scaling": the matmul result
//     is multiplied by the inverse scales of both operands;
//   "Skipping the BAcc accumulator promotion", "DeepSeek FP8 training
//     recipe" > "Mixed-precision accumulation": FP8 multiplicands, FP32
//     accumulation, BF16 (or FP32) result;
//   "DeepSeek FP8 training recipe" > "Block-wise scaling at 128 granularity":
//     block scales applied inside the matmul -- every 128-deep partial sum
//     is scaled by its blocks' factors and added to an FP32 accumulator.
//
// Kernel structure (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: A and B tiles (128 B of K per row, 128-byte
//               swizzle) into a STAGES-deep ring guarded by full/empty
//               mbarriers;
//   warp 1      MMA issuer: one thread issues 4 tcgen05.mma (K = 32 each)
//               per 128-deep stage into a TMEM accumulator and releases the
//               stage with tcgen05.commit;
//   warp 2      TMEM allocation / release;
//   warps 4..   epilogue: tcgen05.ld of the accumulator (thread = row),
//               scale, convert, store to global memory.
// Per-tensor kernel: BM x BN = 128 x 256, two TMEM accumulators (512
// columns) so the epilogue of one tile overlaps the mainloop of the next.
// Block-scaled kernel (fp32 factors): CTA pairs, 256 x 256 tiles, two TMEM
// partial-sum buffers rotated per 128-deep K block; 16 promotion warps per
// CTA add them into FP32 registers.
// Block-scaled kernel (power-of-two factors): CTA pairs, 256 x 256 tiles,
// tcgen05.mma kind::mxf8f6f4.block_scale with the factors as UE8M0 words in
// a TMEM ring written by four factor-writer warps.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/fp8linear.h"
#include "internal.h"
#include "ptx.cuh"

namespace fp8 {

__device__ unsigned int g_device_status = 0;

// Time limit of the single-CTA kernel's epilogue wait for a full accumulator
// (the wait of the epilogue warps, which have nothing asynchronous in flight
// behind them: when it gives up, the producer and MMA threads finish or stop
// at their own bounded waits, drain what they issued, and the kernel returns
// with bit 0 of the status word set).  The library never changes it; the test
// hook fp8_test_set_epilogue_wait_ns() shortens it to make that path run.
__device__ uint64_t g_epilogue_wait_ns = ptx::kWaitTimeoutNs;

namespace {

constexpr int BM = 128;
constexpr int BK = 128;      // bytes = FP8 elements of K per stage
constexpr int UMMA_K = 32;   // K of one kind::f8f6f4 instruction

struct GemmParams {
    int64_t M, N, K;
    int num_m, num_n, num_kb;
    int fa, fb;
    int ga, gb;
    const float* sa;
    const float* sb;
    const __nv_bfloat16* bias;   // nullable: [N], added before the output rounding
    void* D;
    int out;          // FP8_OUT_BF16 / FP8_OUT_F32
    int accumulate;
    int a_mn, b_mn;   // operand stored MN-major ([K x M] / [K x N]); CTA pairs, or 128 x 128 single-CTA tiles
    int group;        // CTA-pair kernel: raster group (M-blocks), see pair_group()
};

// Eight bias values of columns n .. n+7 (n % 8 == 0) as fp32; every lane of
// a warp reads the same 16 bytes, so the load is one broadcast.
__device__ __forceinline__ void load_bias8(float (&b)[8], const __nv_bfloat16* bias, int64_t n) {
    const uint4 v = *reinterpret_cast<const uint4*>(bias + n);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        b[2 * e] = __uint_as_float(w[e] << 16);
        b[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

// Grouped rasterisation: walk GROUP consecutive M-blocks down each N-column
// so that the CTAs resident at one time share A and B panels in L2.  A
// larger group re-reads each B panel from DRAM fewer times (once per group)
// at the cost of more A panels resident at once.
template <int GROUP = 16>
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& m_blk,
                                            int& n_blk) {
    const int per_group = GROUP * num_n;
    const int g = tile / per_group;
    const int first_m = g * GROUP;
    const int gsize = min(num_m - first_m, GROUP);
    const int in_g = tile - g * per_group;
    m_blk = first_m + in_g % gsize;
    n_blk = in_g / gsize;
}

// The same walk with a run-time group size.
__device__ __forceinline__ void tile_coords_g(int tile, int num_m, int num_n, int group,
                                              int& m_blk, int& n_blk) {
    const int per_group = group * num_n;
    const int g = tile / per_group;
    const int first_m = g * group;
    const int gsize = min(num_m - first_m, group);
    const int in_g = tile - g * per_group;
    m_blk = first_m + in_g % gsize;
    n_blk = in_g / gsize;
}

template <int BN, int STAGES>
struct Layout {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + 1024;  // + alignment slack
};

// Raster group of the single-CTA kernel: its producer and its epilogue walk
// the tiles in the same order.
constexpr int kTensorGroup = 8;

// Dequantisation factors of one 32-column chunk, f[j] = fp32(fa * sb(n0 + j)):
// fa is the thread's row factor (sa[m] for per-row A, else sa[0]); sb is per
// column for per-row B (lane j loads column n0 + j, shuffled to all lanes)
// or sb[0].  Warp-collective: every lane of the warp calls it.
__device__ __forceinline__ void chunk_factors(float (&f)[32], float fa, int64_t n0,
                                              const GemmParams& p) {
    if (p.gb == FP8_GRAN_ROW) {
        const int lane = threadIdx.x & 31;
        const float sbv = n0 + lane < p.N ? p.sb[n0 + lane] : 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __fmul_rn(fa, __shfl_sync(0xFFFFFFFFu, sbv, j));
    } else {
        const float a = __fmul_rn(fa, p.sb[0]);
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = a;
    }
}

// Row factor of the A operand for row m (clamped into the matrix).
__device__ __forceinline__ float row_factor(const GemmParams& p, int64_t m) {
    return p.ga == FP8_GRAN_ROW ? p.sa[m < p.M ? m : p.M - 1] : p.sa[0];
}

// Epilogue of one 32-column chunk of an accumulator row: multiply column j
// by f[j], add the bias (if any), then round to bf16 or (optionally) add
// into the FP32 buffer; 16-byte stores.  N % 8 == 0.
__device__ __forceinline__ void store_chunk(const uint32_t (&r)[32], int64_t m, int64_t n0,
                                            const GemmParams& p, const float (&f)[32], bool rmw) {
    if (p.out == FP8_OUT_BF16) {
        __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.D) + m * p.N;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            if (n0 + j < p.N) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(__uint_as_float(r[j + e]), f[j + e]);
                if (p.bias) {
                    float b[8];
                    load_bias8(b, p.bias, n0 + j);
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __fadd_rn(v[e], b[e]);
                }
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                    w[e] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(drow + n0 + j) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.D) + m * p.N + n0);
        // all loads of the chunk first, so that their latencies overlap
        float4 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = (rmw && n0 + 4 * j < p.N) ? dst[j] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (n0 + 4 * j < p.N) {
                float4 v = make_float4(__fmul_rn(__uint_as_float(r[4 * j]), f[4 * j]),
                                       __fmul_rn(__uint_as_float(r[4 * j + 1]), f[4 * j + 1]),
                                       __fmul_rn(__uint_as_float(r[4 * j + 2]), f[4 * j + 2]),
                                       __fmul_rn(__uint_as_float(r[4 * j + 3]), f[4 * j + 3]));
                if (p.bias) {
                    const uint2 bw = *reinterpret_cast<const uint2*>(p.bias + n0 + 4 * j);
                    v.x = __fadd_rn(v.x, __uint_as_float(bw.x << 16));
                    v.y = __fadd_rn(v.y, __uint_as_float(bw.x & 0xFFFF0000u));
                    v.z = __fadd_rn(v.z, __uint_as_float(bw.y << 16));
                    v.w = __fadd_rn(v.w, __uint_as_float(bw.y & 0xFFFF0000u));
                }
                if (rmw) {
                    v.x += o[j].x; v.y += o[j].y; v.z += o[j].z; v.w += o[j].w;
                }
                dst[j] = v;
            }
        }
    }
}

// The FP32 accumulation rows that an epilogue thread will read for a tile:
// pulled into L2 while the tensor cores work, so the read-modify-write hits L2.
__device__ __forceinline__ void prefetch_row(int64_t m, int64_t n0, int width,
                                             const GemmParams& p) {
    if (m >= p.M) return;
    const int64_t cols = p.N - n0 < width ? p.N - n0 : width;
    ptx::prefetch_l2(static_cast<const float*>(p.D) + m * p.N + n0, static_cast<uint32_t>(cols * 4));
}

// Stage one output box of 32 rows x 64 bytes (this thread's row: four 16-byte
// pieces) in `slot` (2 KB of shared memory) with the TMA's 64-byte swizzle --
// piece j of row r at piece j ^ ((r >> 1) & 3), so the 32 rows' writes hit
// distinct banks -- and write it to global memory at (x, y) with a TMA bulk
// store, or, with `add`, a TMA reduce-add (D += box, one FP32 add per element
// performed by the memory system).  Whole-warp call.  The slot is reused, so
// the previous box's store must first have read it.  in_range = false skips
// the store (the box starts past the matrix) but keeps the group count.
__device__ __forceinline__ void emit_box(uint8_t* slot, const uint4 (&piece)[4],
                                         const CUtensorMap* map, int64_t x, int64_t y,
                                         bool in_range, bool add) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) ptx::bulk_wait_group_read<0>();
    __syncwarp();
    uint8_t* row = slot + lane * 64;
    const int swz = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(row + 16 * (j ^ swz)) = piece[j];
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (in_range) {
            if (add)
                ptx::tma_reduce_add_2d(map, ptx::smem_u32(slot), static_cast<int32_t>(x),
                                       static_cast<int32_t>(y));
            else
                ptx::tma_store_2d(map, ptx::smem_u32(slot), static_cast<int32_t>(x),
                                  static_cast<int32_t>(y));
        }
        ptx::bulk_commit_group();
    }
}

// FP32 output of one 32-column accumulator chunk of a warp's 32 rows (first
// row m0, first column n0): v = fp32(acc * f) (+ bias), as two 16-column TMA
// boxes through `slot`, stored or (accumulate) added.  Whole-warp call.
__device__ __forceinline__ void emit_f32_chunk(uint8_t* slot, const uint32_t (&r)[32],
                                               const float (&f)[32], int64_t m0, int64_t n0,
                                               const GemmParams& p, const CUtensorMap* map) {
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __fmul_rn(__uint_as_float(r[e]), f[e]);
    if (p.bias) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            if (n0 + j < p.N) {
                float b[8];
                load_bias8(b, p.bias, n0 + j);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[j + e] = __fadd_rn(v[j + e], b[e]);
            }
        }
    }
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
        uint4 piece[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            piece[j] = make_uint4(__float_as_uint(v[16 * hb + 4 * j]),
                                  __float_as_uint(v[16 * hb + 4 * j + 1]),
                                  __float_as_uint(v[16 * hb + 4 * j + 2]),
                                  __float_as_uint(v[16 * hb + 4 * j + 3]));
        const int64_t x = n0 + 16 * hb;
        emit_box(slot, piece, map, x, m0, m0 < p.M && x < p.N, p.accumulate != 0);
    }
}

// bf16 output of one 32-column accumulator chunk of a warp's 32 rows (first
// row m0, first column n0): v = fp32(acc * f) (+ bias), rounded to bf16, as
// one 32-row x 64-byte TMA box through `slot` (rows past M and columns past N
// are clipped by the copy).  Whole-warp call.
__device__ __forceinline__ void emit_bf16_chunk(uint8_t* slot, const uint32_t (&r)[32],
                                                const float (&f)[32], int64_t m0, int64_t n0,
                                                const GemmParams& p, const CUtensorMap* map) {
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __fmul_rn(__uint_as_float(r[e]), f[e]);
    if (p.bias) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            if (n0 + j < p.N) {
                float b[8];
                load_bias8(b, p.bias, n0 + j);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[j + e] = __fadd_rn(v[j + e], b[e]);
            }
        }
    }
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const uint4 piece[4] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]),
                            make_uint4(w[8], w[9], w[10], w[11]),
                            make_uint4(w[12], w[13], w[14], w[15])};
    emit_box(slot, piece, map, n0, m0, m0 < p.M && n0 < p.N, false);
}

// --------------------------------------------------------- per-tensor kernel

// Single-CTA kernel: 128 x BN tiles, one or (GROUPED) two problems in one
// launch -- the units are the tiles of p, then those of p2, dealt
// round-robin to the CTAs.  An operand is read K-major or (a_mn / b_mn, only
// with BN = 128) MN-major, as the CTA-pair kernel reads it: boxes of
// (128 K bytes, rows) or (128 M/N elements, 128 k).
template <int BN, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(256, 1)
    gemm_tensor_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ GemmParams p,
                       const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ GemmParams p2) {
    ptx::griddep_launch_dependents();   // the next kernel may launch now
    using L = Layout<BN, STAGES>;
    constexpr uint32_t TMEM_COLS = 2 * BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + L::RING_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t1 = p.num_m * p.num_n;
    const int num_units = GROUPED ? t1 + p2.num_m * p2.num_n : t1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 4);
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        if (GROUPED && num_units > t1) {
            ptx::tma_prefetch_desc(&tmA2);
            ptx::tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 2) {
        ptx::tmem_alloc(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    ptx::griddep_wait();   // the previous kernel's results (operands, factors) are visible

    if (warp == 0) {
        if (lane == 0) {
            // producer: the A / B tiles of every K block of this CTA's units
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                const bool second = GROUPED && u >= t1;
                const GemmParams& q = second ? p2 : p;
                const CUtensorMap* ma = second ? &tmA2 : &tmA;
                const CUtensorMap* mb = second ? &tmB2 : &tmB;
                int m_blk, n_blk;
                tile_coords<kTensorGroup>(second ? u - t1 : u, q.num_m, q.num_n, m_blk, n_blk);
                const int ya = m_blk * BM, yb = n_blk * BN;
                for (int kb = 0; kb < q.num_kb; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    uint8_t* sa = ring + stage * L::STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
                    const int kx = kb * BK;
                    ptx::tma_load_2d(sa, ma, &full[stage], q.a_mn ? ya : kx, q.a_mn ? kx : ya);
                    ptx::tma_load_2d(sa + L::A_BYTES, mb, &full[stage], q.b_mn ? yb : kx,
                                     q.b_mn ? kx : yb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // drain: the last copy issued into each slot must have landed
            uint32_t never = 0;
            for (int s = 0; s < STAGES; ++s) {
                if (issued <= s && issued < STAGES) break;
                const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1u);
                ptx::mbar_wait(&full[s], par, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc1 = ptx::idesc_f8f6f4(p.fa, p.fb, BM, BN, p.a_mn, p.b_mn);
            const uint32_t idesc2 = ptx::idesc_f8f6f4(p2.fa, p2.fb, BM, BN, p2.a_mn, p2.b_mn);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                const bool second = GROUPED && u >= t1;
                const int num_kb = second ? p2.num_kb : p.num_kb;
                const uint32_t idesc = second ? idesc2 : idesc1;
                const bool a_mn = (second ? p2.a_mn : p.a_mn) != 0;
                const bool b_mn = (second ? p2.b_mn : p.b_mn) != 0;
                // descriptor advance per MMA of K = 32, in 16-byte units: 32
                // bytes along a K-major row, or 32 rows of 128 bytes MN-major
                const uint32_t a_step = a_mn ? (UMMA_K * 128) >> 4 : UMMA_K >> 4;
                const uint32_t b_step = b_mn ? (UMMA_K * 128) >> 4 : UMMA_K >> 4;
                const uint64_t a_tmpl = a_mn ? ptx::sdesc_mnmajor_sw128(0) : ptx::sdesc_kmajor_sw128(0);
                const uint64_t b_tmpl = b_mn ? ptx::sdesc_mnmajor_sw128(0) : ptx::sdesc_kmajor_sw128(0);
                if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    uint8_t* sa = ring + stage * L::STAGE_BYTES;
                    const uint64_t ad = a_tmpl | ((ptx::smem_u32(sa) & 0x3FFFFu) >> 4);
                    const uint64_t bd = b_tmpl | ((ptx::smem_u32(sa + L::A_BYTES) & 0x3FFFFu) >> 4);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        ptx::mma_f8f6f4(d, ad + k * a_step, bd + k * b_step, idesc, (kb | k) != 0);
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit(&tfull[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every MMA issued by this thread must finish before TMEM is released
            uint32_t never = 0;
            ptx::mma_commit(done);
            ptx::mbar_wait(done, 0, &never);
        }
    } else if (warp >= 4) {
        const int qd = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = qd * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        const uint64_t wait_ns = g_epilogue_wait_ns;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const bool second = GROUPED && u >= t1;
            const GemmParams& q = second ? p2 : p;   // this unit's problem
            const bool rmw = q.out == FP8_OUT_F32 && q.accumulate;
            int m_blk, n_blk;
            tile_coords<kTensorGroup>(second ? u - t1 : u, q.num_m, q.num_n, m_blk, n_blk);
            if (rmw)
                prefetch_row(static_cast<int64_t>(m_blk) * BM + row, static_cast<int64_t>(n_blk) * BN,
                             BN, q);
            bool ok = (lane == 0) ? ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, wait_ns)
                                  : false;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            __syncwarp();
            ptx::tc_fence_after();
            const int64_t m = static_cast<int64_t>(m_blk) * BM + row;
            const float fa = row_factor(q, m);
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
                ptx::tmem_wait_ld();
                const int64_t n0 = static_cast<int64_t>(n_blk) * BN + c * 32;
                float f[32];
                chunk_factors(f, fa, n0, q);
                if (m < q.M) store_chunk(r, m, n0, q, f, rmw);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_device_status, 1u);
}

// ------------------------------------------------------- CTA-pair kernel

// A cluster of two CTAs (on the two SMs of a TPC) computes a 256 x 256 tile
// with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 32):
//   - CTA r loads rows [r*128, r*128+128) of the tile's A panel and of its B
//     panel into its own ring (16 + 16 KiB per stage), so each SM streams
//     half the B bytes that a 128 x 256 single-CTA tile needs;
//   - both CTAs' TMA completions count on the even CTA's `full` barrier, whose
//     MMA thread issues the pair MMAs; each CTA's TMEM receives its 128 rows
//     of the 256 x 256 FP32 accumulator (two accumulators, 512 columns);
//   - MMA completion is multicast to both CTAs' `empty` and `tfull` barriers;
//     both CTAs' epilogue warps arrive on the even CTA's `tempty` barrier, with
//     a relaxed arrive: it only reports that their tcgen05.ld results are in
//     registers, and a cluster-scope release would stall them on a fence.
// GROUPED: a second problem (tmA2, tmB2, p2) shares the launch; without
// it those parameters are ignored and the kernel is the single-problem one.
template <int STAGES, bool GROUPED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ GemmParams p,
                     const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ CUtensorMap tmB2,
                     const __grid_constant__ CUtensorMap tmD2,
                     const __grid_constant__ GemmParams p2) {
    ptx::griddep_launch_dependents();   // the next kernel may launch now
    constexpr int HALF = 128;              // rows of A and of B held by each CTA
    constexpr int TILE = 2 * HALF;         // pair tile: 256 x 256
    constexpr int A_BYTES = HALF * BK, B_BYTES = HALF * BK;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * TILE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = ring + STAGES * STAGE_BYTES;   // FP32 output boxes: 2 KB per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + 4 * 2048);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 8);      // 4 epilogue warps x 2 CTAs
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    // work units: the tiles of problem 1, then those of problem 2 (a second
    // GEMM of the same pass, e.g. the dgrad next to the wgrad; none if
    // p2.num_m == 0), dealt round-robin to the clusters
    const int t1 = p.num_m * p.num_n;
    const int num_units = GROUPED ? t1 + p2.num_m * p2.num_n : t1;
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        if (GROUPED && num_units > t1) {
            ptx::tma_prefetch_desc(&tmA2);
            ptx::tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 2) {
        ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // the peer's barriers exist before any remote arrival
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    ptx::griddep_wait();   // the previous kernel's results (operands, factors) are visible
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                const bool second = GROUPED && u >= t1;
                const GemmParams& q = second ? p2 : p;
                const CUtensorMap* ma = second ? &tmA2 : &tmA;
                const CUtensorMap* mb = second ? &tmB2 : &tmB;
                int m_blk, n_blk;
                tile_coords_g(second ? u - t1 : u, q.num_m, q.num_n, q.group, m_blk, n_blk);
                const int ya = m_blk * TILE + static_cast<int>(rank) * HALF;
                const int yb = n_blk * TILE + static_cast<int>(rank) * HALF;
                const bool a_mn = q.a_mn != 0, b_mn = q.b_mn != 0;
                for (int kb = 0; kb < q.num_kb; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint32_t bar = ptx::cluster_addr(&full[stage], 0);
                    if (leader) ptx::mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    // K-major: box (128 K bytes, 128 rows); MN-major: box
                    // (128 M/N elements, 128 k) -- 16 KB either way
                    const int kx = kb * BK;
                    ptx::tma_load_2d_pair(sa, ma, bar, a_mn ? ya : kx, a_mn ? kx : ya);
                    ptx::tma_load_2d_pair(sa + A_BYTES, mb, bar, b_mn ? yb : kx, b_mn ? kx : yb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            uint32_t never = 0;
            if (leader) {
                // drain: the last copies into each slot (both CTAs' bytes) have landed
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s && issued < STAGES) break;
                    const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1u);
                    ptx::mbar_wait(&full[s], par, &never);
                }
            } else if (!ok) {
                // copies signal the peer's barriers: after an abort, give those in
                // flight a bounded grace period to land before this CTA moves on
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc1 = ptx::idesc_f8f6f4(p.fa, p.fb, TILE, TILE, p.a_mn, p.b_mn);
            const uint32_t idesc2 = ptx::idesc_f8f6f4(p2.fa, p2.fb, TILE, TILE, p2.a_mn, p2.b_mn);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                const bool second = GROUPED && u >= t1;
                const int num_kb = second ? p2.num_kb : p.num_kb;
                const uint32_t idesc = second ? idesc2 : idesc1;
                const bool a_mn = (second ? p2.a_mn : p.a_mn) != 0;
                const bool b_mn = (second ? p2.b_mn : p.b_mn) != 0;
                // descriptor advance per MMA of K = 32, in 16-byte units: 32
                // bytes along a K-major row, or 32 rows of 128 bytes MN-major
                const uint32_t a_step = a_mn ? (UMMA_K * 128) >> 4 : UMMA_K >> 4;
                const uint32_t b_step = b_mn ? (UMMA_K * 128) >> 4 : UMMA_K >> 4;
                // the descriptors' fixed fields; the start address is or-ed in per stage
                const uint64_t a_tmpl = a_mn ? ptx::sdesc_mnmajor_sw128(0) : ptx::sdesc_kmajor_sw128(0);
                const uint64_t b_tmpl = b_mn ? ptx::sdesc_mnmajor_sw128(0) : ptx::sdesc_kmajor_sw128(0);
                if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + acc * TILE;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint64_t ad = a_tmpl | ((ptx::smem_u32(sa) & 0x3FFFFu) >> 4);
                    const uint64_t bd = b_tmpl | ((ptx::smem_u32(sa + A_BYTES) & 0x3FFFFu) >> 4);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        ptx::mma_f8f6f4_pair(d, ad + k * a_step, bd + k * b_step, idesc,
                                             (kb | k) != 0);
                    ptx::mma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit_pair(&tfull[acc], 0x3);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            uint32_t never = 0;
            ptx::mma_commit_pair(done, 0x1);
            ptx::mbar_wait(done, 0, &never);
        }
    } else if (warp >= 4) {
        // 32-row x 64-byte TMA boxes from this warp's 2 KB staging slot: 32
        // bf16 columns stored, or 16 FP32 columns stored or (accumulate) added
        // by the TMA -- no read of D by the SM
        const int qd = warp & 3;
        uint8_t* slot = epi_stage + qd * 2048;
        const GemmParams& p1 = p;
        uint32_t acc = 0, acc_phase = 0;
        for (int u = pair; u < num_units; u += npairs) {
            const bool second = GROUPED && u >= t1;
            const GemmParams& p = second ? p2 : p1;   // this unit's problem
            const CUtensorMap* map = second ? &tmD2 : &tmD;
            const bool f32 = p.out == FP8_OUT_F32;
            int m_blk, n_blk;
            tile_coords_g(second ? u - t1 : u, p.num_m, p.num_n, p.group, m_blk, n_blk);
            const int64_t m0 = static_cast<int64_t>(m_blk) * TILE + rank * HALF + qd * 32;
            const int64_t m = m0 + lane;
            bool ok = (lane == 0) ? ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag) : false;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            __syncwarp();
            ptx::tc_fence_after();
            const float fa = row_factor(p, m);
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + acc * TILE;
#pragma unroll 1
            for (int c = 0; c < TILE / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
                ptx::tmem_wait_ld();
                const int64_t n0 = static_cast<int64_t>(n_blk) * TILE + c * 32;
                float f[32];
                chunk_factors(f, fa, n0, p);
                if (f32) emit_f32_chunk(slot, r, f, m0, n0, p, map);
                else emit_bf16_chunk(slot, r, f, m0, n0, p, map);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_relaxed(ptx::cluster_addr(&tempty[acc], 0));
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) ptx::bulk_wait_group_all();   // every TMA store has completed
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();   // the pair's MMAs, copies and remote arrivals are all done
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_device_status, 1u);
}

// --------------------------------------------------------- block-scaled kernel

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// Block-scaled GEMM with fp32 factors ("Block-wise scaling at 128
// granularity": every 128-deep partial sum is multiplied by its blocks'
// factors before it is added to the FP32 accumulator).
//
// A cluster of two CTAs (the two SMs of a TPC) computes a 256 x TN tile with
// tcgen05.mma.cta_group::2 (M = 256, N = TN, K = 32): CTA r loads rows
// [r*128, r*128+128) of the tile's A panel and rows [r*TN/2, (r+1)*TN/2) of
// its B panel; both CTAs' copies count on the even CTA's `full` barrier,
// whose MMA thread issues the MMAs.  Each 128-deep K block goes to its own
// TMEM buffer (512 / TN buffers of TN columns, rotated), so the MMAs of the
// next blocks run while the promotion warps promote one.  The pair tile
// halves the operand bytes each SM moves through shared memory per FLOP
// against a 128 x TN single-CTA tile.
//   warp 0      TMA producer (one thread);
//   warp 1      MMA issuer (one thread of the even CTA): per K block, waits
//               for a free buffer and a full stage, issues 4 MMAs, commits
//               the stage (`empty`) and the buffer (`tfull`) to both CTAs;
//   warp 2      TMEM allocation (512 columns per CTA);
//   warps 4-    promotion, EPI / 4 per TMEM lane quarter, CW = 4 TN / EPI
//               columns each: per K block, read the buffer (tcgen05.ld),
//               hand it back to the MMA thread (both CTAs' warps arrive on
//               the even CTA's `tempty`), then add partial * s_a(m, kb) *
//               s_b(n, kb) into FP32 registers with packed fma.rn.f32x2.  The
//               factors of the next four K blocks are loaded while the
//               current four are promoted.  At the tile's end the accumulator
//               is rounded (plus the bias) and leaves through 32-row x
//               64-byte TMA boxes: bf16 stores, or FP32 stores / reduce-adds
//               (accumulate).
// Every wait is a blocking try_wait, so that waiting promotion warps do not
// take issue slots from the producer and MMA warps on their sub-partitions.
// COLSCALE: B carries 1x128 scales (one factor per output column and K
// block, the block-wise wgrad); each promotion warp stages its columns'
// factors of four K blocks in shared memory, read back as broadcasts, and its
// rows' factors beside them (the factor products leave no registers for them).
//
// The instance (BpWide): 256 x 256 tiles, so that each MMA is N = 256 (with
// N = 128 the MMAs alone stop at 0.54-0.60 of the tensor core's rate,
// against 0.9 with N = 256).  TMEM then holds two partial-sum buffers, so a
// K block's promotion has to hand its buffer back within the next block's
// MMAs; 16 promotion warps of 64 columns share that work.  The accumulator
// takes 64 registers a thread, so the role warpgroup gives registers back
// with setmaxnreg (32 a thread) and the promotion warps take them (112):
// 4 x 32 x 32 + 16 x 32 x 112 = 61440 = 640 threads x the 96 registers of
// the launch.  Measured against the alternatives (CUDA events, 16384 x
// 18432 x 7168 and 16384 x 7168 x 18432): one 32-column TMEM load at a time (two in flight need 64 more
// registers and spill; 16-column loads were 11% slower); three operand
// stages (four and five were 1.5% and about 5% slower: shared memory comes
// out of L1, where 97% of the promotion warps' factor reads hit); factors
// read at the start of each group of four K blocks rather than one group
// ahead (6% faster: the prefetched values held 8 registers and made the loop
// spill); per-column factor products by packed mul.rn.f32x2 (scalar
// multiplies made the COLSCALE loop 38% slower) and, for COLSCALE, 16-column
// TMEM loads (3% faster there, with fewer spills); 256 x 160 tiles with three
// buffers and 20 promotion warps were 30% slower, and 256 x 128 tiles with
// four buffers and 8 warps (the earlier form) 24% slower (COLSCALE: 9%).
template <int TN_, int EPI_, int STAGES_, int RROLE_, int RPROMO_>
struct BpCfg {
    static constexpr int TN = TN_;
    static constexpr int EPI = EPI_;
    static constexpr int STAGES = STAGES_;
    // registers per thread of the role warpgroup and of the promotion warps
    // after setmaxnreg
    static constexpr int RROLE = RROLE_;
    static constexpr int RPROMO = RPROMO_;
    static constexpr int NBUF = 512 / TN;
    static constexpr int THREADS = (4 + EPI) * 32;
    static constexpr int CW = 4 * TN / EPI;          // columns of one promotion warp
    static constexpr int A_BYTES = 128 * BK;         // this CTA's 128 rows of A
    static constexpr int B_BYTES = (TN / 2) * BK;    // this CTA's half of the TN rows of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // shared memory: operand ring, 2 KB of output staging per promotion
    // warp, per-column and per-row factors (COLSCALE only), barriers,
    // alignment slack
    static constexpr int smem(bool colscale) {
        return STAGES * STAGE_BYTES + EPI * (2048 + (colscale ? 4 * (CW + 32) * 4 : 0)) + 256 +
               1024;
    }
    static_assert(CW == 64, "a warp's columns: one 64-column slice of a 128-column factor "
                            "block, loaded as two 32-column chunks");
    static_assert(4 * 32 * RROLE + EPI * 32 * RPROMO <= THREADS * (65536 / THREADS / 8 * 8),
                  "the register split fits the launch's registers");
};
using BpWide = BpCfg<256, 16, 3, 32, 112>;

// Factors of row r of an operand (gran: FP8_GRAN_TENSOR, 1x128 or 128x128;
// KB blocks per row) for the K blocks kb0 .. kb0+3, 0 past the last block.
// vec: the four are one aligned float4 (KB % 4 == 0, 16-byte aligned array).
__device__ __forceinline__ void block_factors4(float (&f)[4], const float* s, int gran, int64_t r,
                                               int kb0, int KB, bool vec) {
    if (gran == FP8_GRAN_TENSOR) {
        const float v = s[0];
        f[0] = f[1] = f[2] = f[3] = v;
        return;
    }
    if (kb0 >= KB) {
        f[0] = f[1] = f[2] = f[3] = 0.0f;
        return;
    }
    const float* src = s + (gran == FP8_GRAN_1x128 ? r : (r >> 7)) * KB + kb0;
    if (vec) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) f[j] = kb0 + j < KB ? src[j] : 0.0f;
    }
}

// acc[e] += r[2e..2e+1] * f for the NC / 2 packed pairs of NC columns.
template <int NC>
__device__ __forceinline__ void promote_uniform(uint64_t* acc, const uint32_t* r, uint64_t ff) {
#pragma unroll
    for (int e = 0; e < NC / 2; ++e)
        acc[e] = ptx::ffma2(static_cast<uint64_t>(r[2 * e]) | (static_cast<uint64_t>(r[2 * e + 1]) << 32),
                            ff, acc[e]);
}

// acc[e] += r[2e..2e+1] * fp32(fa * cf[2e..2e+1]) for NC columns: per-column
// factors cf (NC floats in shared memory, read as broadcasts).
template <int NC>
__device__ __forceinline__ void promote_columns(uint64_t* acc, const uint32_t* r, float fa,
                                                const float* cf) {
    const uint64_t faa = pack2(fa, fa);
#pragma unroll
    for (int e4 = 0; e4 < NC / 4; ++e4) {
        const float4 c = *reinterpret_cast<const float4*>(cf + 4 * e4);
        const uint64_t f0 = ptx::fmul2(faa, pack2(c.x, c.y));
        const uint64_t f1 = ptx::fmul2(faa, pack2(c.z, c.w));
        acc[2 * e4] = ptx::ffma2(static_cast<uint64_t>(r[4 * e4]) |
                                     (static_cast<uint64_t>(r[4 * e4 + 1]) << 32),
                                 f0, acc[2 * e4]);
        acc[2 * e4 + 1] = ptx::ffma2(static_cast<uint64_t>(r[4 * e4 + 2]) |
                                         (static_cast<uint64_t>(r[4 * e4 + 3]) << 32),
                                     f1, acc[2 * e4 + 1]);
    }
}

// Round one promoted 32-column chunk (16 packed pairs) plus the bias (if
// any) and write it through the warp's staging slot: one bf16 box of 32
// columns, or two FP32 boxes of 16 columns (added to D when accumulating).
// Whole-warp call; m0 is the warp's first row, n0 the chunk's first column.
__device__ __forceinline__ void emit_block_chunk(uint8_t* slot, const uint64_t* acc, int64_t m0,
                                                 int64_t n0, const GemmParams& p,
                                                 const CUtensorMap* map) {
    float v[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        v[2 * e] = __uint_as_float(static_cast<uint32_t>(acc[e]));
        v[2 * e + 1] = __uint_as_float(static_cast<uint32_t>(acc[e] >> 32));
    }
    if (p.bias) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            float b[8];
            load_bias8(b, p.bias, n0 + j);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[j + e] = __fadd_rn(v[j + e], b[e]);
        }
    }
    if (p.out == FP8_OUT_BF16) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const uint4 piece[4] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]),
                                make_uint4(w[8], w[9], w[10], w[11]),
                                make_uint4(w[12], w[13], w[14], w[15])};
        emit_box(slot, piece, map, n0, m0, m0 < p.M, false);
    } else {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint4 piece[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                piece[j] = make_uint4(__float_as_uint(v[16 * hb + 4 * j]),
                                      __float_as_uint(v[16 * hb + 4 * j + 1]),
                                      __float_as_uint(v[16 * hb + 4 * j + 2]),
                                      __float_as_uint(v[16 * hb + 4 * j + 3]));
            emit_box(slot, piece, map, n0 + 16 * hb, m0, m0 < p.M, p.accumulate != 0);
        }
    }
}

template <typename Cfg, bool COLSCALE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    gemm_block_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmD,
                           const __grid_constant__ GemmParams p, int vec_a, int vec_b) {
    ptx::griddep_launch_dependents();   // the next kernel may launch now
    constexpr int STAGES = Cfg::STAGES, NBUF = Cfg::NBUF, EPI = Cfg::EPI;
    constexpr int A_BYTES = Cfg::A_BYTES;
    constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
    constexpr int TN = Cfg::TN;
    constexpr uint32_t TMEM_COLS = 512;   // allocations are powers of two
    static_assert(NBUF * TN <= 512, "the partial-sum buffers fit in TMEM");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = ring + STAGES * STAGE_BYTES;   // output boxes: 2 KB per epilogue warp
    float* colf = reinterpret_cast<float*>(epi_stage + EPI * 2048);   // [warp][4][cols + 32]
    uint64_t* full = reinterpret_cast<uint64_t*>(colf + (COLSCALE ? EPI * 4 * (Cfg::CW + 32) : 0));
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + NBUF;
    uint64_t* done = tempty + NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], 2 * EPI);   // promotion warps of both CTAs
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        ptx::tma_prefetch_desc(&tmD);
    }
    if (warp == 2) {
        ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // the peer's barriers exist before any remote arrival
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    ptx::griddep_wait();   // the previous kernel's results (operands, factors) are visible
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_units = p.num_m * p.num_n;
    const int KB = p.num_kb;

    if (warp < 4) {
    ptx::setmaxnreg_dec<Cfg::RROLE>();   // the whole role warpgroup
    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                int m_blk, n_blk;
                tile_coords_g(u, p.num_m, p.num_n, p.group, m_blk, n_blk);
                const int ya = m_blk * 256 + static_cast<int>(rank) * 128;
                const int yb = n_blk * TN + static_cast<int>(rank) * (TN / 2);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint32_t bar = ptx::cluster_addr(&full[stage], 0);
                    if (leader) ptx::mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    ptx::tma_load_2d_pair(sa, &tmA, bar, kb * BK, ya);
                    ptx::tma_load_2d_pair(sa + A_BYTES, &tmB, bar, kb * BK, yb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            uint32_t never = 0;
            if (leader) {
                // drain: the last copies into each slot (both CTAs' bytes) have landed
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s && issued < STAGES) break;
                    const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1u);
                    ptx::mbar_wait(&full[s], par, &never);
                }
            } else if (!ok) {
                // copies signal the peer's barriers: after an abort, give those in
                // flight a bounded grace period to land before this CTA moves on
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = ptx::idesc_f8f6f4(p.fa, p.fb, 256, TN);
            uint32_t stage = 0, phase = 0, buf = 0, buf_phase = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!ptx::mbar_wait(&tempty[buf], buf_phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(ptx::smem_u32(sa));
                    const uint64_t bd = ptx::sdesc_kmajor_sw128(ptx::smem_u32(sa + A_BYTES));
                    const uint32_t d = tmem_base + buf * TN;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        ptx::mma_f8f6f4_pair(d, ad + (k * UMMA_K >> 4), bd + (k * UMMA_K >> 4),
                                             idesc, k != 0);
                    ptx::mma_commit_pair(&empty[stage], 0x3);
                    ptx::mma_commit_pair(&tfull[buf], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++buf == NBUF) { buf = 0; buf_phase ^= 1u; }
                }
            }
            uint32_t never = 0;
            ptx::mma_commit_pair(done, 0x1);
            ptx::mbar_wait(done, 0, &never);
        }
    }
    } else {
        ptx::setmaxnreg_inc<Cfg::RPROMO>();   // each promotion warpgroup
        constexpr int CW = Cfg::CW;              // columns of this warp
        constexpr int NCH = CW / 32;             // 32-column chunks (COLSCALE factors, stores)
        const int qd = warp & 3;                 // TMEM lane quarter of this warp
        const int h = (warp - 4) >> 2;           // which CW-column slice of the tile
        uint8_t* slot = epi_stage + (warp - 4) * 2048;
        // COLSCALE: the columns' factors [4 K blocks][CW], then the rows'
        // [4 K blocks][32 lanes]
        float* cf = colf + (warp - 4) * 4 * (CW + 32);
        float* rf = cf + 4 * CW;
        const uint32_t lanes = static_cast<uint32_t>(qd * 32) << 16;
        uint32_t buf = 0, buf_phase = 0;
        bool ok = true;
        for (int u = pair; ok && u < num_units; u += npairs) {
            int m_blk, n_blk;
            tile_coords_g(u, p.num_m, p.num_n, p.group, m_blk, n_blk);
            const int64_t m0 = static_cast<int64_t>(m_blk) * 256 + rank * 128 + qd * 32;
            const int64_t m = m0 + lane;
            const int64_t m_safe = m < p.M ? m : p.M - 1;
            const int64_t n0 = static_cast<int64_t>(n_blk) * TN + h * CW;
            // a warp's columns lie all inside or all outside [0, N) (N is a
            // multiple of 128, CW divides 128); outside, its factors are
            // read at column N - 1 and its columns are not stored
            const int64_t nf = n0 < p.N ? n0 : p.N - 1;
            // FP32 accumulator of CW columns, as packed pairs
            uint64_t acc[CW / 2];
#pragma unroll
            for (int e = 0; e < CW / 2; ++e) acc[e] = 0ull;
            for (int kb0 = 0; ok && kb0 < KB; kb0 += 4) {
                // The factors of four K blocks, read at the start of the group
                // (they hit L1; holding the next group's in registers made the
                // loop spill): A per row; B per 128-column block, multiplied
                // into fa here, or (COLSCALE) per column, staged in shared
                // memory for broadcast reads (lane l writes columns n0+32c+l),
                // with the rows' factors beside them (registers are short).
                float fa[4], fb[4];
                block_factors4(fa, p.sa, p.ga, m_safe, kb0, KB, vec_a != 0);
                if (COLSCALE) {
                    __syncwarp();   // the previous group's factors have been read
#pragma unroll
                    for (int j = 0; j < 4; ++j) rf[j * 32 + lane] = fa[j];
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        block_factors4(fb, p.sb, p.gb, nf + (n0 < p.N ? 32 * c + lane : 0), kb0, KB,
                                       vec_b != 0);
#pragma unroll
                        for (int j = 0; j < 4; ++j) cf[j * CW + 32 * c + lane] = fb[j];
                    }
                    __syncwarp();
                } else {
                    block_factors4(fb, p.sb, p.gb, nf, kb0, KB, vec_b != 0);
#pragma unroll
                    for (int j = 0; j < 4; ++j) fa[j] = __fmul_rn(fa[j], fb[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (kb0 + j >= KB) break;
                    ok = (lane == 0) ? ptx::mbar_wait(&tfull[buf], buf_phase, abort_flag) : false;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok) break;
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint32_t ta = tmem_base + lanes + buf * TN + h * CW;
                    // The warp's 64 columns as two 32-column loads, one at a
                    // time (the accumulator takes most of the registers); the
                    // buffer goes back once the last has landed.  Measured:
                    // overlapping the second half's loads with the first
                    // half's promotion (16-column loads) spilled or ran 4-46%
                    // slower.  COLSCALE, whose factor products need more
                    // registers, loads 16 columns at a time (3% faster).
                    if constexpr (COLSCALE) {
                        const float faj = rf[j * 32 + lane];
                        const float* cfj = cf + j * CW;
                        uint32_t r[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            ptx::tmem_ld_32x32b_x16(ta + 16 * c, r);
                            ptx::tmem_wait_ld();
                            if (c == 3) {
                                ptx::tc_fence_before();
                                __syncwarp();
                                if (lane == 0)
                                    ptx::mbar_arrive_cluster_relaxed(ptx::cluster_addr(&tempty[buf], 0));
                            }
                            promote_columns<16>(acc + 8 * c, r, faj, cfj + 16 * c);
                        }
                    } else {
                        const uint64_t ff = pack2(fa[j], fa[j]);
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(ta, r);
                        ptx::tmem_wait_ld();
                        promote_uniform<32>(acc, r, ff);
                        ptx::tmem_ld_32x32b_x32(ta + 32, r);
                        ptx::tmem_wait_ld();
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            ptx::mbar_arrive_cluster_relaxed(ptx::cluster_addr(&tempty[buf], 0));
                        promote_uniform<32>(acc + 16, r, ff);
                    }
                    if (++buf == NBUF) { buf = 0; buf_phase ^= 1u; }
                }
            }
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                if (n0 < p.N) emit_block_chunk(slot, acc + 16 * c, m0, n0 + 32 * c, p, &tmD);
        }
        if (lane == 0) ptx::bulk_wait_group_all();   // every TMA store has completed
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();   // the pair's MMAs, copies and remote arrivals are all done
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_device_status, 1u);
}

// ------------------------------------------ block-scaled kernel, power-of-two factors

// With power-of-two factors the block scales go into the tensor core itself
// (tcgen05.mma kind::mxf8f6f4.block_scale, one UE8M0 factor per 32 elements
// of K): each 1x128 or 128x128 factor is given to the four 32-deep K steps of
// its 128-deep block, so the products are the same terms as "Block-wise
// scaling at 128 granularity" computes, and the accumulator stays in TMEM for
// the whole K loop as with per-tensor scales -- nothing is promoted per K
// block.
//
// Factor words: a 32-bit TMEM word holds four UE8M0 bytes and each MMA picks
// one of them (the instruction descriptor's factor byte), so one word serves
// four K blocks (byte j: K block 4w + j of the slot).  A ring slot holds four
// words per row, i.e. the factors of 16 K blocks; the MMA selects the word by
// the TMEM address it passes (A: slot + 4w, B: slot + 16 + 8w).
//   A, row r of the CTA's 128:      lane r, column slot + 4w + r/32
//   B, row n of the tile's 256:     column slot + 16 + 8w + n/32 of lane
//                                   32q + n%32, for every lane quarter q
//                                   (each quarter reads its own copy)
//
// CTA pair (cluster of 2), 256 x 256 tiles, one TMEM accumulator (256
// columns) plus the factor ring in the other 256 columns.
//   warp 0      TMA producer (as the per-tensor pair kernel);
//   warp 1      MMA issuer (even CTA): per K block, waits for the operand
//               stage (and, every 16 K blocks, for a factor slot), issues 4
//               block-scaled MMAs, then releases the stage (and the slot
//               after its 16th K block) with tcgen05.commit;
//   warp 2      TMEM allocation;
//   warps 4-7   factor writers: per slot, load the fp32 factors coalesced
//               (4 lanes per row, 16 K blocks of a row in one 64-byte
//               segment), convert them to UE8M0 words, exchange them
//               through shared memory, and tcgen05.st each lane quarter's
//               A words and copy of the B words into the slot;
//   warps 8-15  epilogue, 2 per lane quarter (128 columns each): read the
//               accumulator, hand it back to the MMA as soon as it is in
//               registers, then round and write each 32-row x 64-byte box to
//               a shared-memory staging slot in the TMA's 64-byte swizzled
//               layout and store it with a TMA bulk store -- or, for an
//               accumulating FP32 output, a TMA reduce-add (D += box, one
//               FP32 add per element, as a read-modify-write would do).
//               Row-per-thread global stores (32 rows per instruction) held
//               up the next tile's MMA issue.
constexpr int kMxStages = 6;
constexpr int kMxSfSlots = 4;
constexpr int kMxEpiWarps = 8;
constexpr int kMxThreads = (8 + kMxEpiWarps) * 32;
constexpr int kMxStageA = 4 * 136;   // words per buffer: [word][128 rows + pad]
constexpr int kMxStageB = 4 * 264;   //                   [word][256 rows + pad]
constexpr int kMxEpiStage = 2048;     // bytes of output staging per epilogue warp: one box
constexpr int kMxSmemBytes = kMxStages * 2 * 128 * BK + kMxEpiWarps * kMxEpiStage +
                             2 * (kMxStageA + kMxStageB) * 4 + 512 + 1024;

// Factors of row r (of an operand with `rows` rows) for the K blocks
// kb0 .. kb0+3; 1.0 outside the matrix and past the last K block.  vec: the
// four are one aligned float4 (KB % 4 == 0 and a 16-byte aligned array).
__device__ __forceinline__ void mx_load4(float (&f)[4], const float* s, int gran, int64_t r,
                                         int64_t rows, int kb0, int KB, bool vec) {
    if (r >= rows || kb0 >= KB) {
        f[0] = f[1] = f[2] = f[3] = 1.0f;
        return;
    }
    const float* src = s + (gran == FP8_GRAN_1x128 ? r : (r >> 7)) * KB + kb0;
    if (vec) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) f[j] = kb0 + j < KB ? src[j] : 1.0f;
    }
}

// TMEM factor word of four power-of-two factors: byte j is the UE8M0 code
// of f[j] -- its biased fp32 exponent; mantissa bits are ignored, and 2^-127
// or less gives 0.
__device__ __forceinline__ uint32_t ue8m0_word(const float (&f)[4]) {
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) w |= ((__float_as_uint(f[j]) >> 23) & 0xFFu) << (8 * j);
    return w;
}

// One 32-column accumulator chunk (FP32 bits) plus the bias (if any) as 16
// bf16 pairs, rounded to nearest even -- the same values store_chunk writes
// with unit factors.  Columns past N are packed but never stored.
__device__ __forceinline__ void pack_bf16_chunk(uint32_t (&pk)[16], const uint32_t (&r)[32],
                                                int64_t n0, const GemmParams& p) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[j + e]);
        if (p.bias && n0 + j < p.N) {
            float b[8];
            load_bias8(b, p.bias, n0 + j);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __fadd_rn(v[e], b[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            pk[j / 2 + e] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
}

template <int STAGES, int SFS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMxThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ GemmParams p, int vec_a, int vec_b) {
    ptx::griddep_launch_dependents();   // the next kernel may launch now
    constexpr int HALF = 128;              // rows of A and of B held by each CTA
    constexpr int TILE = 2 * HALF;         // pair tile: 256 x 256
    constexpr int A_BYTES = HALF * BK, B_BYTES = HALF * BK;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t SF_COL0 = TILE;     // factor ring after the accumulator
    constexpr uint32_t SF_SLOT = 48;       // columns per slot: A at +0..15, B at +16..47
    constexpr int KPS = 16;                // K blocks per slot
    static_assert(SF_COL0 + SFS * SF_SLOT <= TMEM_COLS, "factor ring exceeds TMEM");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = ring + STAGES * STAGE_BYTES;   // [8 warps][2048 B], 1024-aligned
    uint32_t* stage_a = reinterpret_cast<uint32_t*>(epi_stage + kMxEpiWarps * kMxEpiStage);  // [2][4][136]
    uint32_t* stage_b = stage_a + 2 * kMxStageA;                                  // [2][4][264]
    uint64_t* full = reinterpret_cast<uint64_t*>(stage_b + 2 * kMxStageB);
    uint64_t* empty = full + STAGES;
    uint64_t* sf_full = empty + STAGES;
    uint64_t* sf_empty = sf_full + SFS;
    uint64_t* tfull = sf_empty + SFS;
    uint64_t* tempty = tfull + 1;
    uint64_t* done = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < SFS; ++s) {
            ptx::mbar_init(&sf_full[s], 8);   // 4 writer warps x 2 CTAs
            ptx::mbar_init(&sf_empty[s], 1);
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 2 * kMxEpiWarps);
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        ptx::tma_prefetch_desc(&tmD);
    }
    if (warp == 2) {
        ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // the peer's barriers exist before any remote arrival
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    ptx::griddep_wait();   // the previous kernel's results (operands, factors) are visible
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_units = p.num_m * p.num_n;
    const int num_slots = (p.num_kb + KPS - 1) / KPS;   // factor slots per tile

    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                int m_blk, n_blk;
                tile_coords_g(u, p.num_m, p.num_n, p.group, m_blk, n_blk);
                const int ya = m_blk * TILE + static_cast<int>(rank) * HALF;
                const int yb = n_blk * TILE + static_cast<int>(rank) * HALF;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint32_t bar = ptx::cluster_addr(&full[stage], 0);
                    if (leader) ptx::mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    ptx::tma_load_2d_pair(sa, &tmA, bar, kb * BK, ya);
                    ptx::tma_load_2d_pair(sa + A_BYTES, &tmB, bar, kb * BK, yb);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            uint32_t never = 0;
            if (leader) {
                // drain: the last copies into each slot (both CTAs' bytes) have landed
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s && issued < STAGES) break;
                    const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1u);
                    ptx::mbar_wait(&full[s], par, &never);
                }
            } else if (!ok) {
                // copies signal the peer's barriers: after an abort, give those in
                // flight a bounded grace period to land before this CTA moves on
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // factor byte j (K block 4w + j of the slot's word w) in both bytes fields
            const uint32_t idesc0 = ptx::idesc_mxf8f6f4(p.fa, p.fb, TILE, TILE, 0, 0);
            uint32_t stage = 0, phase = 0, sfs = 0, sf_phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                if (!ptx::mbar_wait(tempty, acc_phase ^ 1u, abort_flag)) break;
                ptx::tc_fence_after();
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    if ((kb % KPS) == 0 &&
                        !ptx::mbar_wait(&sf_full[sfs], sf_phase, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(ptx::smem_u32(sa));
                    const uint64_t bd = ptx::sdesc_kmajor_sw128(ptx::smem_u32(sa + A_BYTES));
                    const uint32_t w = static_cast<uint32_t>(kb % KPS) >> 2;
                    const uint32_t byte = static_cast<uint32_t>(kb) & 3u;
                    const uint32_t sfa = tmem_base + SF_COL0 + sfs * SF_SLOT + 4 * w;
                    const uint32_t sfb = tmem_base + SF_COL0 + sfs * SF_SLOT + 16 + 8 * w;
                    const uint32_t id = idesc0 | (byte << 4) | (byte << 29);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        ptx::mma_mxf8f6f4_pair(tmem_base, ad + (k * UMMA_K >> 4),
                                               bd + (k * UMMA_K >> 4), id, sfa, sfb, (kb | k) != 0);
                    ptx::mma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if ((kb % KPS) == KPS - 1 || kb == p.num_kb - 1) {   // the slot's last K block
                        ptx::mma_commit_pair(&sf_empty[sfs], 0x3);
                        if (++sfs == SFS) { sfs = 0; sf_phase ^= 1u; }
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(tfull, 0x3);
                acc_phase ^= 1u;
            }
            uint32_t never = 0;
            ptx::mma_commit_pair(done, 0x1);
            ptx::mbar_wait(done, 0, &never);
        }
    } else if (warp >= 4 && warp < 8) {
        // factor writers: warp 4 + q owns TMEM lanes 32q .. 32q+31.  Loads use
        // 4 lanes per row (lane = 4 * row + K quarter), 8 rows per instruction:
        // warp q loads A rows 32q + 8i + lane/4 (i < 4) and B rows
        // 64q + 8i + lane/4 (i < 8), K blocks 16s + 4 (lane % 4) .. + 3.
        const int q = warp & 3;
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        const int rsub = lane >> 2, kq = lane & 3;
        uint32_t sfs = 0, sf_phase = 0, buf = 0;
        // after a failed wait this warp keeps meeting the writers' named barrier
        // (so that the other three cannot wait on it forever) but does nothing else
        bool live = true;
        for (int u = pair; u < num_units; u += npairs) {
            int m_blk, n_blk;
            tile_coords_g(u, p.num_m, p.num_n, p.group, m_blk, n_blk);
            const int64_t a0 = static_cast<int64_t>(m_blk) * TILE + rank * HALF;
            const int64_t b0 = static_cast<int64_t>(n_blk) * TILE;
            for (int s2 = 0; s2 < num_slots; ++s2) {
                uint32_t* sta = stage_a + buf * kMxStageA;
                uint32_t* stb = stage_b + buf * kMxStageB;
                if (live) {
                    const int kb0 = KPS * s2 + 4 * kq;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = q * 32 + 8 * i + rsub;
                        float f[4];
                        mx_load4(f, p.sa, p.ga, a0 + row, p.M, kb0, p.num_kb, vec_a != 0);
                        sta[kq * 136 + row] = ue8m0_word(f);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = q * 64 + 8 * i + rsub;
                        float f[4];
                        mx_load4(f, p.sb, p.gb, b0 + row, p.N, kb0, p.num_kb, vec_b != 0);
                        stb[kq * 264 + row] = ue8m0_word(f);
                    }
                }
                ptx::named_bar_sync(1, 128);   // the slot's words of all four warps are staged
                if (live) {
                    // A: word w at column 4w + q of this quarter's lanes (the other
                    // columns of these lanes are not read)
                    uint32_t wa[16], wb[32];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t v = sta[w * 136 + q * 32 + lane];
#pragma unroll
                        for (int j = 0; j < 4; ++j) wa[4 * w + j] = j == q ? v : 0u;
                    }
#pragma unroll
                    for (int w = 0; w < 4; ++w)
#pragma unroll
                        for (int c = 0; c < 8; ++c) wb[8 * w + c] = stb[w * 264 + 32 * c + lane];
                    bool ok = (lane == 0) ? ptx::mbar_wait(&sf_empty[sfs], sf_phase ^ 1u, abort_flag)
                                          : false;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (ok) {
                        ptx::tc_fence_after();
                        const uint32_t col = tmem_base + lanes + SF_COL0 + sfs * SF_SLOT;
                        ptx::tmem_st_32x32b_x16(col, wa);
                        ptx::tmem_st_32x32b_x32(col + 16, wb);
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster(ptx::cluster_addr(&sf_full[sfs], 0));
                    } else {
                        live = false;
                    }
                }
                if (++sfs == SFS) { sfs = 0; sf_phase ^= 1u; }
                buf ^= 1u;
            }
        }
    } else if (warp >= 8) {
        // epilogue warp: 32 rows (lane quarter q) x 128 columns (half h) of the
        // CTA's 128 x 256 accumulator.  Output boxes are 32 rows x 64 bytes
        // (32 bf16 or 16 FP32 columns), staged with the TMA's 64-byte swizzle:
        // 16-byte piece j of row r at piece j ^ ((r >> 1) & 3).
        const int q = warp & 3, h = (warp - 8) >> 2;
        uint8_t* stg = epi_stage + (warp - 8) * kMxEpiStage;
        const bool f32 = p.out == FP8_OUT_F32;
        const bool add = f32 && p.accumulate;
        float ones[32];   // unit factors: the block scales are applied in the MMA
#pragma unroll
        for (int j = 0; j < 32; ++j) ones[j] = 1.0f;
        uint32_t acc_phase = 0;
        for (int u = pair; u < num_units; u += npairs) {
            int m_blk, n_blk;
            tile_coords_g(u, p.num_m, p.num_n, p.group, m_blk, n_blk);
            const int64_t m0 = static_cast<int64_t>(m_blk) * TILE + rank * HALF + q * 32;
            const int64_t n0 = static_cast<int64_t>(n_blk) * TILE + h * 128;
            bool ok = (lane == 0) ? ptx::mbar_wait(tfull, acc_phase, abort_flag) : false;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            __syncwarp();
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
            // one staged 32-row x 64-byte box to global memory at column x
            auto emit = [&](const uint4 (&piece)[4], int64_t x) {
                emit_box(stg, piece, &tmD, x, m0, m0 < p.M && x < p.N, add);
            };
            if (!f32) {
                // read and pack the 128 columns first, hand the accumulator back,
                // then stage and store
                uint32_t pk[4][16];
#pragma unroll
                for (int c = 0; c < 4; c += 2) {
                    uint32_t r0[32], r1[32];
                    ptx::tmem_ld_32x32b_x32(tbase + c * 32, r0);
                    ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, r1);
                    ptx::tmem_wait_ld();
                    if (c == 2) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster_relaxed(ptx::cluster_addr(tempty, 0));
                    }
                    pack_bf16_chunk(pk[c], r0, n0 + c * 32, p);
                    pack_bf16_chunk(pk[c + 1], r1, n0 + (c + 1) * 32, p);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 piece[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        piece[j] = make_uint4(pk[c][4 * j], pk[c][4 * j + 1], pk[c][4 * j + 2],
                                              pk[c][4 * j + 3]);
                    emit(piece, n0 + c * 32);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; c += 2) {
                    uint32_t r[2][32];
                    ptx::tmem_ld_32x32b_x32(tbase + c * 32, r[0]);
                    ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, r[1]);
                    ptx::tmem_wait_ld();
                    if (c == 2) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster_relaxed(ptx::cluster_addr(tempty, 0));
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        emit_f32_chunk(stg, r[i], ones, m0, n0 + (c + i) * 32, p, &tmD);
                }
            }
            acc_phase ^= 1u;
        }
        if (lane == 0) ptx::bulk_wait_group_all();   // every store has completed
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();   // the pair's MMAs, copies, factor stores and remote arrivals are done
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_device_status, 1u);
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of a K-contiguous FP8 matrix [rows x K]: boxes of 128 bytes of K
// by box_rows rows, 128-byte swizzle, zero fill outside the matrix.
int make_kmajor_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K,
                    uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld]",
                         static_cast<int>(r), static_cast<long long>(rows),
                         static_cast<long long>(K));
    return FP8_OK;
}

// Tensor map of an MN-contiguous FP8 matrix stored [K x MN] (the transpose of
// a K-major operand): boxes of 128 elements of MN by BK rows of K, 128-byte
// swizzle, zero fill outside the matrix.
int make_mnmajor_map(CUtensorMap* map, const void* ptr, int64_t MN, int64_t K) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(MN), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(MN)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(BK)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld]",
                         static_cast<int>(r), static_cast<long long>(K),
                         static_cast<long long>(MN));
    return FP8_OK;
}

}  // namespace

int make_bf16_box_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols,
                      uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for bf16 [%lld x %lld]",
                         static_cast<int>(r), static_cast<long long>(rows),
                         static_cast<long long>(cols));
    return FP8_OK;
}

namespace {

// Tensor map of the output D [M x N] (bf16 or FP32, row-major) for TMA stores
// of boxes of 32 rows x 64 bytes (32 bf16 or 16 FP32 columns) with the
// 64-byte swizzle.
int make_store_map(CUtensorMap* map, void* ptr, int64_t M, int64_t N, int out) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const bool f32 = out == FP8_OUT_F32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {f32 ? 16u : 32u, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for output [%lld x %lld]",
                         static_cast<int>(r), static_cast<long long>(M),
                         static_cast<long long>(N));
    return FP8_OK;
}

constexpr int kTensorBN = 256, kTensorStages = 4;
// Column tiles of the single-CTA kernel for problems whose 128-row tiles fit
// in one wave: 64 columns where those fit, else 128.
constexpr int kSmallBN = 128, kTinyBN = 64;
constexpr int kPairStages = 6;
constexpr int kPairSmemBytes = kPairStages * 2 * 128 * BK + 4 * 2048 + 256 + 1024;
// Problems with at least this many rows use the CTA-pair kernel.
constexpr int64_t kPairMinRows = 256;

template <typename Kernel>
int ensure_smem(Kernel k, int bytes, int kernel_id) {
    static std::mutex mu;
    static bool done[64][16] = {};   // [device][kernel id]: every GEMM kernel has this one type
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    const bool cached = dev >= 0 && dev < 64;   // other devices: set it on every call
    std::lock_guard<std::mutex> lock(mu);
    if (cached && done[dev][kernel_id]) return FP8_OK;
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return set_error(FP8_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    if (cached) done[dev][kernel_id] = true;
    return FP8_OK;
}

// How many 2-CTA clusters of the pair kernel fit on the device at once (the
// persistent grid size); cached per device.
int pair_clusters(const void* func, int kernel_id, int threads, int smem) {
    static std::mutex mu;
    static int cache[64][5] = {};   // [device][kernel id]: 0 single, 1 grouped pair kernel,
                                    // 2 power-of-two block kernel, 3 / 4 fp32-factor block
                                    // kernel (row / column factors on B)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    int uncached = 0;                            // devices past the table: computed per call
    std::lock_guard<std::mutex> lock(mu);
    int& c = (dev >= 0 && dev < 64) ? cache[dev][kernel_id] : uncached;
    if (c == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = num_sms() / 2;
        }
        c = n;
    }
    return c;
}

}  // namespace

int num_sms() {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    int n = dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// D[m][n] (+)= bias[n] for a GEMM with K = 0 (grid-stride over M x N).
__global__ void bias_rows_kernel(const __nv_bfloat16* __restrict__ bias, int64_t M, int64_t N,
                                 void* D, int out, int rmw) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const int64_t n_all = M * N;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_all;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float b = __bfloat162float(bias[i % N]);
        if (out == FP8_OUT_BF16) static_cast<__nv_bfloat16*>(D)[i] = __float2bfloat16_rn(b);
        else static_cast<float*>(D)[i] = rmw ? static_cast<float*>(D)[i] + b : b;
    }
}

namespace {

// Raster group of a CTA-pair problem: the group's A panels (GROUP blocks of
// 256 rows by K bytes) are reused by every N-block of the sweep, so they
// should stay in L2 (129 MB) next to the B panels in flight: at most 64 MB of
// them, between 4 and 16 blocks.  Measured on the Llama-2 step GEMMs, 16 beat
// 8 and 4 where the panels fit; with K = 28672 a group of 16 (117 MB) was
// re-read from DRAM about once per wave.
int pair_group(int64_t K) {
    const int64_t panel = 256 * K;
    int g = 16;
    while (g > 4 && g * panel > (int64_t(64) << 20)) g >>= 1;
    return g;
}

// Block-scaled GEMM with power-of-two factors on the CTA-pair block-scaled
// MMA kernel (ga, gb: FP8_GRAN_1x128 / FP8_GRAN_128x128, flag removed; K > 0).
int launch_gemm_mx(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                   int64_t K, int ga, const float* sa, int gb, const float* sb, const void* bias,
                   void* D, int out, int accumulate, cudaStream_t stream) {
    GemmParams p;
    p.M = M; p.N = N; p.K = K;
    p.num_m = static_cast<int>((M + 255) / 256);
    p.num_n = static_cast<int>((N + 255) / 256);
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    p.fa = fa; p.fb = fb; p.ga = ga; p.gb = gb; p.sa = sa; p.sb = sb;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.D = D; p.out = out; p.accumulate = accumulate;
    p.a_mn = p.b_mn = 0;
    p.group = pair_group(K);
    CUtensorMap tmA, tmB, tmD;
    int st = make_kmajor_map(&tmA, A, M, K, BM);
    if (st != FP8_OK) return st;
    if ((st = make_kmajor_map(&tmB, B, N, K, 128)) != FP8_OK) return st;
    if ((st = make_store_map(&tmD, D, M, N, out)) != FP8_OK) return st;
    auto k = gemm_mx_kernel<kMxStages, kMxSfSlots>;
    if ((st = ensure_smem(k, kMxSmemBytes, 5)) != FP8_OK) return st;
    const int64_t tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    const int64_t clusters =
        pair_clusters(reinterpret_cast<const void*>(k), 2, kMxThreads, kMxSmemBytes);
    const int grid = static_cast<int>(2 * (tiles < clusters ? tiles : clusters));
    // factors of four K blocks as one float4: rows of a multiple of 4 floats, aligned arrays
    const int vec_a = p.num_kb % 4 == 0 && (reinterpret_cast<uintptr_t>(sa) & 15u) == 0;
    const int vec_b = p.num_kb % 4 == 0 && (reinterpret_cast<uintptr_t>(sb) & 15u) == 0;
    launch_pdl(k, dim3(grid), dim3(kMxThreads), kMxSmemBytes, stream, tmA, tmB, tmD, p, vec_a, vec_b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

template <typename C, bool COLSCALE>
int launch_block_cfg(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                     int64_t K, int ga, const float* sa, int gb, const float* sb,
                     const void* bias, void* D, int out, int accumulate, cudaStream_t stream) {
    GemmParams p;
    p.M = M; p.N = N; p.K = K;
    p.num_m = static_cast<int>((M + 255) / 256);
    p.num_n = static_cast<int>((N + C::TN - 1) / C::TN);
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    p.fa = fa; p.fb = fb; p.ga = ga; p.gb = gb; p.sa = sa; p.sb = sb;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.D = D; p.out = out; p.accumulate = accumulate;
    p.a_mn = p.b_mn = 0;
    p.group = pair_group(K);
    CUtensorMap tmA, tmB, tmD;
    int st = make_kmajor_map(&tmA, A, M, K, 128);
    if (st != FP8_OK) return st;
    if ((st = make_kmajor_map(&tmB, B, N, K, C::TN / 2)) != FP8_OK) return st;
    if ((st = make_store_map(&tmD, D, M, N, out)) != FP8_OK) return st;
    auto k = gemm_block_pair_kernel<C, COLSCALE>;
    constexpr int SMEM = C::smem(COLSCALE);
    if ((st = ensure_smem(k, SMEM, COLSCALE ? 3 : 1)) != FP8_OK) return st;
    const int64_t tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    const int64_t clusters = pair_clusters(reinterpret_cast<const void*>(k), COLSCALE ? 4 : 3,
                                           C::THREADS, SMEM);
    const int grid = static_cast<int>(2 * (tiles < clusters ? tiles : clusters));
    // factors of four K blocks as one float4: rows of a multiple of 4 floats, aligned arrays
    const int vec_a = p.num_kb % 4 == 0 && (reinterpret_cast<uintptr_t>(sa) & 15u) == 0;
    const int vec_b = p.num_kb % 4 == 0 && (reinterpret_cast<uintptr_t>(sb) & 15u) == 0;
    launch_pdl(k, dim3(grid), dim3(C::THREADS), SMEM, stream, tmA, tmB, tmD, p, vec_a, vec_b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

// Block-scaled GEMM with fp32 factors (at least one operand with 1x128 or
// 128x128 scales; K > 0) on the CTA-pair promotion kernel (256 x 256 tiles),
// with the per-column factor path when B has 1x128 scales.
int launch_gemm_block(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                      int64_t K, int ga, const float* sa, int gb, const float* sb,
                      const void* bias, void* D, int out, int accumulate, cudaStream_t stream) {
    const bool colscale = gb == FP8_GRAN_1x128;
    return colscale ? launch_block_cfg<BpWide, true>(A, fa, B, fb, M, N, K, ga, sa, gb, sb, bias, D,
                                                     out, accumulate, stream)
                    : launch_block_cfg<BpWide, false>(A, fa, B, fb, M, N, K, ga, sa, gb, sb, bias, D,
                                                      out, accumulate, stream);
}

}  // namespace

namespace {

// Column tile of the single-CTA kernel when an M x N problem's 128-row tiles
// fit in one wave (at most one CTA per SM): 64 where those fit and both
// operands are K-major, else 128 (which also reads MN-major operands); 0
// when neither fits.  Eight or four CTAs per 256 x 256 pair tile, each with
// an eighth or a quarter of its MMAs and epilogue: a small layer's GEMMs,
// where latency is the cost.
int one_wave_bn(int64_t M, int64_t N, bool mn_major) {
    const int64_t sms = num_sms(), rows = (M + BM - 1) / BM;
    if (!mn_major && rows * ((N + kTinyBN - 1) / kTinyBN) <= sms) return kTinyBN;
    if (rows * ((N + kSmallBN - 1) / kSmallBN) <= sms) return kSmallBN;
    return 0;
}

// Launch of the single-CTA kernel with BN-column tiles: problem p1 (and,
// GROUPED, p2 in the same launch; 128-column tiles only).
template <bool GROUPED>
int launch_tensor(int BN, int grid, cudaStream_t stream, const CUtensorMap& a1,
                  const CUtensorMap& b1, const GemmParams& p1, const CUtensorMap& a2,
                  const CUtensorMap& b2, const GemmParams& p2) {
    int st;
    if (GROUPED || BN == kSmallBN) {
        using L = Layout<kSmallBN, kTensorStages>;
        auto k = gemm_tensor_kernel<kSmallBN, kTensorStages, GROUPED>;
        if ((st = ensure_smem(k, L::SMEM_BYTES, GROUPED ? 8 : 6)) != FP8_OK) return st;
        launch_pdl(k, dim3(grid), dim3(256), L::SMEM_BYTES, stream, a1, b1, p1, a2, b2, p2);
    } else if (BN == kTinyBN) {
        using L = Layout<kTinyBN, kTensorStages>;
        auto k = gemm_tensor_kernel<kTinyBN, kTensorStages, false>;
        if ((st = ensure_smem(k, L::SMEM_BYTES, 7)) != FP8_OK) return st;
        launch_pdl(k, dim3(grid), dim3(256), L::SMEM_BYTES, stream, a1, b1, p1, a2, b2, p2);
    } else {
        using L = Layout<kTensorBN, kTensorStages>;
        auto k = gemm_tensor_kernel<kTensorBN, kTensorStages, false>;
        if ((st = ensure_smem(k, L::SMEM_BYTES, 0)) != FP8_OK) return st;
        launch_pdl(k, dim3(grid), dim3(256), L::SMEM_BYTES, stream, a1, b1, p1, a2, b2, p2);
    }
    return FP8_OK;
}

}  // namespace

int launch_gemm(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
                int64_t K, int ga, const float* sa, int gb, const float* sb, const void* bias,
                void* D, int out, int accumulate, cudaStream_t stream, int layout) {
    if (M == 0 || N == 0) return FP8_OK;
    const bool a_mn = (layout & FP8_LAYOUT_A_KM) != 0, b_mn = (layout & FP8_LAYOUT_B_KN) != 0;
    // power-of-two block factors on both operands: the block-scaled MMA
    const bool pow2 = (ga & FP8_SCALE_POW2) && (gb & FP8_SCALE_POW2);
    ga &= ~FP8_SCALE_POW2;
    gb &= ~FP8_SCALE_POW2;
    if (K == 0 && bias) {   // an empty sum: D (+)= bias
        const int64_t n = M * N;
        const int64_t blocks = (n + 255) / 256;
        launch_pdl(bias_rows_kernel, dim3(static_cast<unsigned>(blocks < 65535 * 16 ? blocks : 65535 * 16)), dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(bias), M, N, D, out,
                                        out == FP8_OUT_F32 && accumulate);
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? FP8_OK
                                : set_error(FP8_ERR_CUDA, "bias launch: %s", cudaGetErrorString(e));
    }
    if (K == 0) {
        if (out == FP8_OUT_F32 && accumulate) return FP8_OK;
        const size_t bytes = static_cast<size_t>(M) * N * (out == FP8_OUT_F32 ? 4 : 2);
        const cudaError_t e = cudaMemsetAsync(D, 0, bytes, stream);
        return e == cudaSuccess ? FP8_OK
                                : set_error(FP8_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    }
    const bool block = ga == FP8_GRAN_1x128 || ga == FP8_GRAN_128x128 || gb == FP8_GRAN_1x128 ||
                       gb == FP8_GRAN_128x128;
    const bool mx = pow2 && (ga == FP8_GRAN_1x128 || ga == FP8_GRAN_128x128) &&
                    (gb == FP8_GRAN_1x128 || gb == FP8_GRAN_128x128);
    if (mx) return launch_gemm_mx(A, fa, B, fb, M, N, K, ga, sa, gb, sb, bias, D, out, accumulate,
                                  stream);
    if (block)
        return launch_gemm_block(A, fa, B, fb, M, N, K, ga, sa, gb, sb, bias, D, out, accumulate,
                                 stream);
    // per-tensor and per-row scales.  A problem whose 128-row tiles fit in
    // one wave (at most one CTA per SM) runs on the single-CTA kernel (see
    // one_wave_bn); otherwise CTA pairs for every problem of at least 256 rows
    // or with an MN-major operand, and the single-CTA kernel with 128 x 256
    // tiles for the rest (K-major, M < 256; rows past M are zero-filled and
    // not stored)
    const int one_bn = one_wave_bn(M, N, a_mn || b_mn);
    const bool pair = !one_bn && (M >= kPairMinRows || a_mn || b_mn);
    const int BN = one_bn ? one_bn : kTensorBN;
    const int TM = pair ? 256 : BM;   // rows of C per tile
    GemmParams p;
    p.M = M; p.N = N; p.K = K;
    p.num_m = static_cast<int>((M + TM - 1) / TM);
    p.num_n = static_cast<int>((N + BN - 1) / BN);
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    p.fa = fa; p.fb = fb; p.ga = ga; p.gb = gb; p.sa = sa; p.sb = sb;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.D = D; p.out = out; p.accumulate = accumulate;
    p.a_mn = a_mn; p.b_mn = b_mn;
    p.group = pair_group(K);

    CUtensorMap tmA, tmB;
    int st = a_mn ? make_mnmajor_map(&tmA, A, M, K) : make_kmajor_map(&tmA, A, M, K, BM);
    if (st != FP8_OK) return st;
    st = b_mn ? make_mnmajor_map(&tmB, B, N, K) : make_kmajor_map(&tmB, B, N, K, pair ? 128 : BN);
    if (st != FP8_OK) return st;

    const int64_t tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    const int grid = static_cast<int>(tiles < num_sms() ? tiles : num_sms());
    if (pair) {
        CUtensorMap tmD;
        if ((st = make_store_map(&tmD, D, M, N, out)) != FP8_OK) return st;
        auto k = gemm_pair_kernel<kPairStages, false>;
        if ((st = ensure_smem(k, kPairSmemBytes, 2)) != FP8_OK) return st;
        const int64_t clusters =
            pair_clusters(reinterpret_cast<const void*>(k), 0, 256, kPairSmemBytes);
        const int pgrid = static_cast<int>(2 * (tiles < clusters ? tiles : clusters));
        GemmParams none{};
        launch_pdl(k, dim3(pgrid), dim3(256), kPairSmemBytes, stream, tmA, tmB, tmD, p, tmA, tmB, tmD, none);
    } else if ((st = launch_tensor<false>(BN, grid, stream, tmA, tmB, p, tmA, tmB, p)) != FP8_OK) {
        return st;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

namespace {

// A problem the CTA-pair kernel takes: per-tensor or per-row scales, at least
// 256 rows or an MN-major operand, a nonempty K.
bool pair_eligible(const GemmArgs& g) {
    const int ga = g.ga & ~FP8_SCALE_POW2, gb = g.gb & ~FP8_SCALE_POW2;
    const bool block = ga == FP8_GRAN_1x128 || ga == FP8_GRAN_128x128 ||
                       gb == FP8_GRAN_1x128 || gb == FP8_GRAN_128x128;
    return !block && (g.M >= kPairMinRows || g.layout != FP8_LAYOUT_TN) && g.N > 0 && g.K > 0 &&
           !g.bias;
}

int pair_params(const GemmArgs& g, GemmParams& p, CUtensorMap& tmA, CUtensorMap& tmB,
                CUtensorMap& tmD) {
    p = GemmParams{};
    p.M = g.M; p.N = g.N; p.K = g.K;
    p.num_m = static_cast<int>((g.M + 255) / 256);
    p.num_n = static_cast<int>((g.N + kTensorBN - 1) / kTensorBN);
    p.num_kb = static_cast<int>((g.K + BK - 1) / BK);
    p.fa = g.fa; p.fb = g.fb; p.ga = g.ga; p.gb = g.gb; p.sa = g.sa; p.sb = g.sb;
    p.bias = static_cast<const __nv_bfloat16*>(g.bias);
    p.D = g.D; p.out = g.out; p.accumulate = g.accumulate;
    p.a_mn = (g.layout & FP8_LAYOUT_A_KM) != 0;
    p.b_mn = (g.layout & FP8_LAYOUT_B_KN) != 0;
    p.group = pair_group(g.K);
    int st = p.a_mn ? make_mnmajor_map(&tmA, g.A, g.M, g.K) : make_kmajor_map(&tmA, g.A, g.M, g.K, BM);
    if (st != FP8_OK) return st;
    st = p.b_mn ? make_mnmajor_map(&tmB, g.B, g.N, g.K) : make_kmajor_map(&tmB, g.B, g.N, g.K, 128);
    if (st != FP8_OK) return st;
    return make_store_map(&tmD, g.D, g.M, g.N, g.out);
}

// Parameters and tensor maps of one problem for the single-CTA kernel with
// BN-column tiles (MN-major operands need BN = 128).
int tensor_params(const GemmArgs& g, int BN, GemmParams& p, CUtensorMap& tmA, CUtensorMap& tmB) {
    p = GemmParams{};
    p.M = g.M; p.N = g.N; p.K = g.K;
    p.num_m = static_cast<int>((g.M + BM - 1) / BM);
    p.num_n = static_cast<int>((g.N + BN - 1) / BN);
    p.num_kb = static_cast<int>((g.K + BK - 1) / BK);
    p.fa = g.fa; p.fb = g.fb; p.ga = g.ga; p.gb = g.gb; p.sa = g.sa; p.sb = g.sb;
    p.bias = static_cast<const __nv_bfloat16*>(g.bias);
    p.D = g.D; p.out = g.out; p.accumulate = g.accumulate;
    p.a_mn = (g.layout & FP8_LAYOUT_A_KM) != 0;
    p.b_mn = (g.layout & FP8_LAYOUT_B_KN) != 0;
    int st = p.a_mn ? make_mnmajor_map(&tmA, g.A, g.M, g.K) : make_kmajor_map(&tmA, g.A, g.M, g.K, BM);
    if (st != FP8_OK) return st;
    return p.b_mn ? make_mnmajor_map(&tmB, g.B, g.N, g.K) : make_kmajor_map(&tmB, g.B, g.N, g.K, BN);
}

// Two problems that one launch of the single-CTA kernel takes: per-tensor or
// per-row scales, nonempty, no bias, and their 128 x 128 tiles together in
// one wave (a small layer's dgrad and wgrad).
bool one_wave_group(const GemmArgs& g1, const GemmArgs& g2) {
    auto ok = [](const GemmArgs& g) {
        const int ga = g.ga & ~FP8_SCALE_POW2, gb = g.gb & ~FP8_SCALE_POW2;
        const bool block = ga == FP8_GRAN_1x128 || ga == FP8_GRAN_128x128 ||
                           gb == FP8_GRAN_1x128 || gb == FP8_GRAN_128x128;
        return !block && g.M > 0 && g.N > 0 && g.K > 0 && !g.bias;
    };
    auto tiles = [](const GemmArgs& g) {
        return ((g.M + BM - 1) / BM) * ((g.N + kSmallBN - 1) / kSmallBN);
    };
    return ok(g1) && ok(g2) && tiles(g1) + tiles(g2) <= num_sms();
}

}  // namespace

int launch_gemm_group(const GemmArgs& g1, const GemmArgs& g2, cudaStream_t stream) {
    if (one_wave_group(g1, g2)) {
        GemmParams p1, p2;
        CUtensorMap a1, b1, a2, b2;
        int st = tensor_params(g1, kSmallBN, p1, a1, b1);
        if (st == FP8_OK) st = tensor_params(g2, kSmallBN, p2, a2, b2);
        if (st != FP8_OK) return st;
        const int units = p1.num_m * p1.num_n + p2.num_m * p2.num_n;
        if ((st = launch_tensor<true>(kSmallBN, units, stream, a1, b1, p1, a2, b2, p2)) != FP8_OK)
            return st;
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? FP8_OK
                                : set_error(FP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    }
    if (!pair_eligible(g1) || !pair_eligible(g2)) {
        int st = launch_gemm(g1.A, g1.fa, g1.B, g1.fb, g1.M, g1.N, g1.K, g1.ga, g1.sa, g1.gb,
                             g1.sb, g1.bias, g1.D, g1.out, g1.accumulate, stream, g1.layout);
        if (st != FP8_OK) return st;
        return launch_gemm(g2.A, g2.fa, g2.B, g2.fb, g2.M, g2.N, g2.K, g2.ga, g2.sa, g2.gb,
                           g2.sb, g2.bias, g2.D, g2.out, g2.accumulate, stream, g2.layout);
    }
    GemmParams p1, p2;
    CUtensorMap a1, b1, d1, a2, b2, d2;
    int st = pair_params(g1, p1, a1, b1, d1);
    if (st == FP8_OK) st = pair_params(g2, p2, a2, b2, d2);
    if (st != FP8_OK) return st;
    // the deeper problem's tiles first, so the last round holds the cheaper tiles
    const bool swap = p2.num_kb > p1.num_kb;
    auto k = gemm_pair_kernel<kPairStages, true>;
    if ((st = ensure_smem(k, kPairSmemBytes, 4)) != FP8_OK) return st;
    const int64_t units = static_cast<int64_t>(p1.num_m) * p1.num_n +
                          static_cast<int64_t>(p2.num_m) * p2.num_n;
    const int64_t clusters = pair_clusters(reinterpret_cast<const void*>(k), 1, 256, kPairSmemBytes);
    const int grid = static_cast<int>(2 * (units < clusters ? units : clusters));
    if (swap) launch_pdl(k, dim3(grid), dim3(256), kPairSmemBytes, stream, a2, b2, d2, p2, a1, b1, d1, p1);
    else launch_pdl(k, dim3(grid), dim3(256), kPairSmemBytes, stream, a1, b1, d1, p1, a2, b2, d2, p2);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FP8_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

unsigned* device_status_word() {
    // looked up once per CUDA context (the module, and the word, are loaded
    // per context) and kept under the context's unique ID
    static std::mutex mu;
    static std::vector<std::pair<unsigned long long, unsigned*>> cache;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (id != 0)
        for (const auto& e : cache)
            if (e.first == id) return e.second;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    const unsigned long long id_now = id != 0 ? id : current_context_id();
    if (id_now != 0) cache.emplace_back(id_now, static_cast<unsigned*>(p));
    return static_cast<unsigned*>(p);
}

int set_epilogue_wait_ns(uint64_t ns) {
    const cudaError_t e = cudaMemcpyToSymbol(g_epilogue_wait_ns, &ns, sizeof(ns));
    if (e != cudaSuccess)
        return set_error(FP8_ERR_CUDA, "setting the epilogue wait limit: %s", cudaGetErrorString(e));
    return FP8_OK;
}

int read_device_status(unsigned* status, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return set_error(FP8_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned));
    if (e != cudaSuccess)
        return set_error(FP8_ERR_CUDA, "reading device status: %s", cudaGetErrorString(e));
    if (clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned));
        if (e != cudaSuccess)
            return set_error(FP8_ERR_CUDA, "clearing device status: %s", cudaGetErrorString(e));
    }
    return FP8_OK;
}

}  // namespace fp8
