// quantize.cu -- the memory-bound half of the scaled FP8 linear: amax
// reduction, scale update and the bf16 -> FP8 casts (per-tensor, with an
// optional fused transpose and fused amax; 1x128 and 128x128 block-wise).
//
// Method ("Mixed Precision LLM Training: The Complete Guide"):
//   "Transformer Engine internals" > "Per-tensor scaling": q = fp8(x * s)
//     with s chosen so that max|x| lands at the top of the FP8 range;
//   "Delayed scaling" / "History-based scaling": s comes from the max over
//     an amax history and is applied one step late;
//   "DeepSeek FP8 training recipe" > "Block-wise scaling at 128
//     granularity": one scale per 1x128 row segment or 128x128 tile.
//
// Every kernel streams bf16 in 16-byte vectors and writes FP8 in 8- or
// 16-byte vectors.  amax is an integer max over |bf16| bit patterns
// (sign bit cleared), reduced with warp max-reductions and one atomicMax
// per CTA on the fp32 bit pattern, which orders like the value for
// non-negative floats: the result is exact and independent of order.
#include <cfloat>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8 {
namespace {

constexpr int kThreads = 256;

template <int FMT>
struct Fp8Traits;
template <>
struct Fp8Traits<0> {
    static constexpr __nv_fp8_interpretation_t kind = __NV_E4M3;
    static constexpr float max_finite = 448.0f;
};
template <>
struct Fp8Traits<1> {
    static constexpr __nv_fp8_interpretation_t kind = __NV_E5M2;
    static constexpr float max_finite = 57344.0f;
};

// Two packed bf16 (element 0 in the low half) times s, cast to two FP8
// codes (element 0 in the low byte), saturating, round to nearest even.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(uint32_t w, float s) {
    const float lo = __fmul_rn(__uint_as_float(w << 16), s);
    const float hi = __fmul_rn(__uint_as_float(w & 0xFFFF0000u), s);
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, Fp8Traits<FMT>::kind));
}

// Four bf16 (two words) -> four FP8 codes in one word.
template <int FMT>
__device__ __forceinline__ uint32_t cvt4(uint32_t w0, uint32_t w1, float s) {
    return cvt2<FMT>(w0, s) | (cvt2<FMT>(w1, s) << 16);
}

// Dashboard counters of one cast ("Numerical-failure taxonomy" > "A
// diagnostic dashboard"): `under` counts nonzero inputs whose code is +-0,
// `sat` inputs whose scaled value exceeds the largest finite value.
struct CastCounts {
    uint32_t under = 0, sat = 0;
};

template <int FMT>
__device__ __forceinline__ uint32_t cvt2c(uint32_t w, float s, CastCounts& c) {
    const float lo = __fmul_rn(__uint_as_float(w << 16), s);
    const float hi = __fmul_rn(__uint_as_float(w & 0xFFFF0000u), s);
    const uint32_t pair = static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, Fp8Traits<FMT>::kind));
    c.sat += (fabsf(lo) > Fp8Traits<FMT>::max_finite) + (fabsf(hi) > Fp8Traits<FMT>::max_finite);
    c.under += ((w & 0x7FFFu) != 0 && (pair & 0x7Fu) == 0) +
               ((w & 0x7FFF0000u) != 0 && (pair & 0x7F00u) == 0);
    return pair;
}

// cvt4 with or without counting.
template <int FMT, bool COUNT>
__device__ __forceinline__ uint32_t cvt4x(uint32_t w0, uint32_t w1, float s, CastCounts& c) {
    if (COUNT) return cvt2c<FMT>(w0, s, c) | (cvt2c<FMT>(w1, s, c) << 16);
    return cvt4<FMT>(w0, w1, s);
}

// CTA-wide sum of the counters, added to counts[0..1] with one atomic each.
__device__ __forceinline__ void cta_counts_commit(const CastCounts& c, unsigned long long* counts) {
    __shared__ uint32_t part[2][kThreads / 32];
    const uint32_t u = __reduce_add_sync(0xFFFFFFFFu, c.under);
    const uint32_t v = __reduce_add_sync(0xFFFFFFFFu, c.sat);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        part[0][warp] = u;
        part[1][warp] = v;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = static_cast<int>(blockDim.x >> 5);
        unsigned long long a = lane < nw ? part[0][lane] : 0u, b = lane < nw ? part[1][lane] : 0u;
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
        }
        if (lane == 0) {
            if (a) atomicAdd(&counts[0], a);
            if (b) atomicAdd(&counts[1], b);
        }
    }
}

// ------------------------------------------------------ stochastic rounding
//
// "Mixed Precision LLM Training: The Complete Guide", "Stochastic rounding":
// round up or down at random with the probability set by the remainder, so
// the cast is unbiased.  The random bits come from Philox-4x32-10 (Salmon et
// al., "Parallel random numbers: as easy as 1, 2, 3", SC'11), a counter-based
// generator: element i of a row-major tensor takes word (i mod 4) of
// Philox(counter = (i/4, offset), key = seed), so any thread can draw any
// element's bits without state and the result does not depend on the launch.

struct SrKey {
    uint32_t k0, k1, o0, o1;  // key (seed) and the upper counter words (offset)
};

// The key schedule (the key of each of the ten rounds), computed once per
// thread, and the offset words.
struct SrSched {
    uint32_t k0[10], k1[10], o0, o1;
};

// The key of a launch: the one passed by value, or (seed, counter) read
// from device memory when key_dev is set.
__device__ __forceinline__ SrKey sr_key_of(const SrKey& k, const unsigned long long* key_dev) {
    if (!key_dev) return k;
    const unsigned long long seed = key_dev[0], ctr = key_dev[1];
    return SrKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32),
                 static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32)};
}

__device__ __forceinline__ SrSched sr_sched(const SrKey& k) {
    SrSched s;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        s.k0[r] = k.k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
        s.k1[r] = k.k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    s.o0 = k.o0;
    s.o1 = k.o1;
    return s;
}

// Philox-4x32-10 of counter (lo32(group), hi32(group), o0, o1): ten rounds
// of two 32 x 32 -> 64-bit products (multipliers 0xD2511F53, 0xCD9E8D57)
// whose halves are crossed and XORed with the other counter words and the
// round key.
__device__ __forceinline__ uint4 sr_bits(const SrSched& k, uint64_t group) {
    uint4 c = make_uint4(static_cast<uint32_t>(group), static_cast<uint32_t>(group >> 32), k.o0, k.o1);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = c.x * 0xD2511F53u, hi0 = __umulhi(c.x, 0xD2511F53u);
        const uint32_t lo1 = c.z * 0xCD9E8D57u, hi1 = __umulhi(c.z, 0xCD9E8D57u);
        c = make_uint4(hi1 ^ c.y ^ k.k0[r], lo1, hi0 ^ c.w ^ k.k1[r], lo0);
    }
    return c;
}

// Stochastic rounding of one fp32 value onto the FP8 grid, driven by the
// uniform 32-bit word r.  With f the remainder below the FP8 grid spacing as
// a fraction of that spacing, the magnitude rounds up iff r < floor(f * 2^32).
// The decision is taken by adding ~r (= 2^32 - 1 - r), aligned below the
// kept bits, and truncating: the sum carries into the kept bits exactly when
// r < floor(f * 2^32).  The result is an fp32 value that lies on the FP8 grid
// (or is beyond the largest finite value, +-Inf or NaN), so the saturating
// round-to-nearest conversion that follows is exact.
//  * normal FP8 range, finite: f has 20 (E4M3) or 21 (E5M2) bits, so the add
//    acts on the fp32 bit pattern itself (a mantissa overflow carries into
//    the exponent, never into the sign) and the low bits are then cleared;
//  * below the smallest normal: the 24-bit significand, shifted to fixed
//    point with 32 fraction bits on the subnormal grid, plus ~r, gives the
//    number of grid steps;
//  * +-Inf and NaN pass through (the conversion saturates / yields NaN).
template <int FMT>
__device__ __forceinline__ float sr_round(float v, uint32_t r) {
    constexpr int kMant = FMT == 0 ? 3 : 2, kBias = FMT == 0 ? 7 : 15, kEmin = 1 - kBias;
    constexpr int kShift = 23 - kMant;
    constexpr uint32_t kNormMin = static_cast<uint32_t>(127 + kEmin) << 23;   // 2^emin
    constexpr uint32_t kLow = (1u << kShift) - 1u;
    const uint32_t u = __float_as_uint(v), a = u & 0x7FFFFFFFu;
    if (a - kNormMin < 0x7F800000u - kNormMin)                 // normal range, finite
        return __uint_as_float((u + (kLow - (r >> (32 - kShift)))) & ~kLow);
    if (a >= 0x7F800000u) return v;
    const uint32_t ex = a >> 23;
    const uint32_t sig = ex ? ((a & 0x7FFFFFu) | 0x800000u) : a;
    // grid exponent minus the significand's exponent: >= 24 - kMant
    const int sh = min(kEmin - kMant + 150 - static_cast<int>(max(ex, 1u)), 63);
    const uint64_t t = (static_cast<uint64_t>(sig) << 32) >> sh;
    const uint32_t steps = static_cast<uint32_t>((t + static_cast<uint64_t>(~r)) >> 32);
    const float m = __fmul_rn(__uint2float_rn(steps), __uint_as_float(static_cast<uint32_t>(127 + kEmin - kMant) << 23));
    return __uint_as_float(__float_as_uint(m) | (u & 0x80000000u));
}

// One fp32 value to its stochastically rounded FP8 code.
template <int FMT>
__device__ __forceinline__ uint32_t sr_code(float v, uint32_t r) {
    const float t = sr_round<FMT>(v, r);
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(t, 0.0f), __NV_SATFINITE, Fp8Traits<FMT>::kind)) & 0xFFu;
}

// Four consecutive bf16 (two words) times s to four codes, stochastically
// rounded with the four words of r.
template <int FMT>
__device__ __forceinline__ uint32_t sr4(uint32_t w0, uint32_t w1, float s, uint4 r) {
    const float t0 = sr_round<FMT>(__fmul_rn(__uint_as_float(w0 << 16), s), r.x);
    const float t1 = sr_round<FMT>(__fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), s), r.y);
    const float t2 = sr_round<FMT>(__fmul_rn(__uint_as_float(w1 << 16), s), r.z);
    const float t3 = sr_round<FMT>(__fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), s), r.w);
    const uint32_t lo = static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(t0, t1), __NV_SATFINITE, Fp8Traits<FMT>::kind));
    const uint32_t hi = static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(t2, t3), __NV_SATFINITE, Fp8Traits<FMT>::kind));
    return lo | (hi << 16);
}

// The four codes of elements 4*group .. 4*group+3: round to nearest even
// (with or without counters) or, with SR, stochastically.
template <int FMT, bool COUNT, bool SR>
__device__ __forceinline__ uint32_t cast4(uint32_t w0, uint32_t w1, float s, CastCounts& c,
                                          const SrSched& k, uint64_t group) {
    if constexpr (SR) {
        static_assert(!COUNT, "stochastic rounding has no counters");
        return sr4<FMT>(w0, w1, s, sr_bits(k, group));
    } else {
        return cvt4x<FMT, COUNT>(w0, w1, s, c);
    }
}

// 16 consecutive bf16 (two 16-byte vectors) starting at element 16*v.
template <int FMT, bool COUNT, bool SR>
__device__ __forceinline__ uint4 cast16(const uint4& a, const uint4& b, float s, CastCounts& c,
                                        const SrSched& k, uint64_t v) {
    return make_uint4(cast4<FMT, COUNT, SR>(a.x, a.y, s, c, k, 4 * v),
                      cast4<FMT, COUNT, SR>(a.z, a.w, s, c, k, 4 * v + 1),
                      cast4<FMT, COUNT, SR>(b.x, b.y, s, c, k, 4 * v + 2),
                      cast4<FMT, COUNT, SR>(b.z, b.w, s, c, k, 4 * v + 3));
}

// Running per-halfword max of |bf16| bit patterns.
__device__ __forceinline__ uint32_t absmax2(uint32_t m, uint32_t w) {
    return __vmaxu2(m, w & 0x7FFF7FFFu);
}

__device__ __forceinline__ uint32_t absmax_vec(uint32_t m, const uint4& v) {
    m = absmax2(m, v.x);
    m = absmax2(m, v.y);
    m = absmax2(m, v.z);
    return absmax2(m, v.w);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Reduce a per-thread |bf16| max (packed or not) over the CTA and raise
// *amax_bits to it (fp32 bit pattern = bf16 bits << 16).
__device__ __forceinline__ void cta_amax_commit(uint32_t m2, unsigned* amax_bits) {
    __shared__ uint32_t warp_max[kThreads / 32];
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = lane < (int)(blockDim.x >> 5) ? warp_max[lane] : 0u;
        v = __reduce_max_sync(0xFFFFFFFFu, v);
        if (lane == 0 && v != 0) atomicMax(amax_bits, v << 16);
    }
}

// Scale of one block from its amax: fp8_max / amax, clamped to the normal
// fp32 range, optionally rounded down to a power of two; 1 for an all-zero
// or non-finite block.
template <int FMT>
__device__ __forceinline__ float block_scale(float amax, int pow2) {
    if (!(amax > 0.0f) || !isfinite(amax)) return 1.0f;
    float s = __fdiv_rn(Fp8Traits<FMT>::max_finite, amax);
    if (!(s <= FLT_MAX)) s = FLT_MAX;
    if (s < FLT_MIN) s = FLT_MIN;
    if (pow2) s = __uint_as_float(__float_as_uint(s) & 0xFF800000u);
    return s;
}

// ------------------------------------------------------------------ amax

// The amax of up to two tensors in one launch (the X and W of a forward
// pass): CTAs [0, ctas0) walk job 0 grid-stride, the rest job 1.
struct AmaxJob {
    const uint4* x;        // the 8-element vectors
    int64_t nvec;
    const uint16_t* tail;  // the last tail_n (< 8) elements
    int tail_n;
    unsigned* amax_bits;
};

__global__ void __launch_bounds__(kThreads) amax_kernel(AmaxJob j0, AmaxJob j1, int ctas0) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const bool second = static_cast<int>(blockIdx.x) >= ctas0;
    const AmaxJob& j = second ? j1 : j0;
    const uint4* __restrict__ x = j.x;
    const int64_t nvec = j.nvec;
    const int64_t cta = second ? blockIdx.x - ctas0 : blockIdx.x;
    const int64_t nctas = second ? gridDim.x - ctas0 : ctas0;
    uint32_t m = 0;
    const int64_t stride = nctas * blockDim.x;
    int64_t i = cta * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 a = ldg_stream(x + i), b = ldg_stream(x + i + stride);
        const uint4 c = ldg_stream(x + i + 2 * stride), d = ldg_stream(x + i + 3 * stride);
        m = absmax_vec(m, a);
        m = absmax_vec(m, b);
        m = absmax_vec(m, c);
        m = absmax_vec(m, d);
    }
    for (; i < nvec; i += stride) m = absmax_vec(m, ldg_stream(x + i));
    if (cta == 0 && threadIdx.x < j.tail_n) m = max(m, (uint32_t)(j.tail[threadIdx.x] & 0x7FFFu));
    cta_amax_commit(m, j.amax_bits);
}

// ---------------------------------------------------------- scale update

// The scale of an effective amax 0 < a < inf: fp8_max / a * 2^-margin,
// clamped to [FLT_MIN, FLT_MAX], optionally rounded down to a power of two.
__device__ __forceinline__ float scale_from_amax(float fmax, float a, int margin, int pow2) {
    float s = __fdiv_rn(fmax, a);
    s = __fmul_rn(s, __uint_as_float(static_cast<uint32_t>(127 - margin) << 23));
    if (!(s <= FLT_MAX)) s = FLT_MAX;
    if (s < FLT_MIN) s = FLT_MIN;
    if (pow2) s = __uint_as_float(__float_as_uint(s) & 0xFF800000u);
    return s;
}

// The scale a cast with a fused dynamic update uses (every thread), given the
// role's amax a, and the role's state update (the thread with `writer` set).
__device__ __forceinline__ float dynamic_scale_of(const ScaleUpd& u, float fmax, float a,
                                                  bool writer) {
    const bool ok = a > 0.0f && isfinite(a);
    const float s = ok ? scale_from_amax(fmax, a, u.margin, u.pow2) : *u.scale;
    if (writer) {
        u.history[*u.pos] = a;
        *u.pos = 0;   // history length 1
        if (!isfinite(a) && u.status) atomicOr(u.status, 2u);
        if (ok) {
            *u.scale = s;
            *u.scale_inv = __fdiv_rn(1.0f, s);
        }
        if (u.saved) *u.saved = *u.scale_inv;
    }
    return s;
}

// The same with the amax that an amax pass left in the role's slot.
__device__ __forceinline__ float fused_dynamic_scale(const ScaleUpd& u, float fmax, bool writer) {
    return dynamic_scale_of(u, fmax, *u.amax, writer);
}

// One warp per role.  history[pos] = amax; pos = (pos + 1) % H;
// a = max(history) or amax; if 0 < a < inf: s = fp8_max / a * 2^-margin,
// clamped to [FLT_MIN, FLT_MAX], optionally rounded down to 2^k; scale = s,
// scale_inv = 1 / s.  Otherwise scale and scale_inv are left unchanged.
// `saved` (nullable) receives scale_inv[r] as it was before the update
// (save_after = 0) or after it (save_after = 1): the dequantisation factor of
// the operand that the same pass cast with the old or the new scale.
__global__ void update_scale_kernel(const float* __restrict__ amax, float* __restrict__ history,
                                    int32_t* __restrict__ pos, int H, int algo, float fmax,
                                    int margin, int pow2, float* __restrict__ scale,
                                    float* __restrict__ scale_inv, float* __restrict__ saved,
                                    int save_after, unsigned* status) {
    // (tiny kernel: the next one may launch once the kernel before this one
    // has completed, not earlier, so a chain of launches cannot run ahead of
    // a large kernel)
    ptx::griddep_wait();   // the previous kernel's results are visible
    ptx::griddep_launch_dependents();
    const int r = blockIdx.x, lane = threadIdx.x;
    float* hist = history + static_cast<int64_t>(r) * H;
    const float a = amax[r];
    const int p = pos[r];
    // NaN-dominant max over the history with the new value in slot p
    float eff = -INFINITY;
    if (algo == 0) {
        for (int i = lane; i < H; i += 32) {
            const float h = (i == p) ? a : hist[i];
            if (isnan(h) || h > eff) eff = h;
        }
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, eff, off);
            if (isnan(o) || o > eff) eff = o;
        }
    } else {
        eff = a;
    }
    __syncwarp();
    if (lane == 0) {
        if (saved && !save_after) saved[r] = scale_inv[r];
        hist[p] = a;
        pos[r] = (p + 1 == H) ? 0 : p + 1;
        // a NaN or Inf in the tensor (or still in the history): the scale
        // stays, and the device status word records it ("Numerical-failure
        // taxonomy": catch NaN / Inf at the first step that sees them)
        if (!isfinite(eff) && status) atomicOr(status, 2u);
        if (eff > 0.0f && isfinite(eff)) {
            const float s = scale_from_amax(fmax, eff, margin, pow2);
            scale[r] = s;
            scale_inv[r] = __fdiv_rn(1.0f, s);
        }
        if (saved && save_after) saved[r] = scale_inv[r];
    }
}

// ------------------------------------------------------- per-tensor cast

// Flat cast, 16 elements (32 B in, 16 B out) per thread per step: the
// stochastic-rounding form (the round-to-nearest casts use the chunked
// kernel below).
template <int FMT, bool AMAX, bool COUNT, bool SR>
__global__ void __launch_bounds__(kThreads)
    quantize_flat_kernel(const uint4* __restrict__ x, int64_t n16, const uint16_t* __restrict__ xt,
                         int tail_n, const float* __restrict__ scale_p, uint4* __restrict__ q,
                         uint8_t* __restrict__ qtail, unsigned* amax_bits,
                         unsigned long long* counts, SrKey sr_key,
                         const unsigned long long* key_dev) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const float s = *scale_p;
    const SrSched key = sr_sched(sr_key_of(sr_key, SR ? key_dev : nullptr));
    uint32_t m = 0;
    CastCounts cc;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + stride < n16; i += 2 * stride) {
        const uint4 a0 = ldg_stream(x + 2 * i), b0 = ldg_stream(x + 2 * i + 1);
        const uint4 a1 = ldg_stream(x + 2 * (i + stride)), b1 = ldg_stream(x + 2 * (i + stride) + 1);
        if (AMAX) m = absmax_vec(absmax_vec(absmax_vec(absmax_vec(m, a0), b0), a1), b1);
        q[i] = cast16<FMT, COUNT, SR>(a0, b0, s, cc, key, i);
        q[i + stride] = cast16<FMT, COUNT, SR>(a1, b1, s, cc, key, i + stride);
    }
    for (; i < n16; i += stride) {
        const uint4 a = ldg_stream(x + 2 * i), b = ldg_stream(x + 2 * i + 1);
        if (AMAX) m = absmax_vec(absmax_vec(m, a), b);
        q[i] = cast16<FMT, COUNT, SR>(a, b, s, cc, key, i);
    }
    if (blockIdx.x == 0 && threadIdx.x < tail_n) {
        const uint32_t w = xt[threadIdx.x];
        if (AMAX) m = max(m, w & 0x7FFFu);
        uint32_t code;
        if constexpr (SR) {
            const uint64_t e = static_cast<uint64_t>(n16) * 16 + threadIdx.x;
            const uint4 r = sr_bits(key, e >> 2);
            const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
            code = sr_code<FMT>(__fmul_rn(__uint_as_float(w << 16), s), rw[e & 3]);
        } else {
            code = COUNT ? cvt2c<FMT>(w & 0xFFFFu, s, cc) : cvt2<FMT>(w, s);
        }
        qtail[threadIdx.x] = static_cast<uint8_t>(code & 0xFFu);
    }
    if (AMAX) cta_amax_commit(m, amax_bits);
    if (COUNT) cta_counts_commit(cc, counts);
}

// Round-to-nearest cast without a transpose, one chunk per CTA: each thread
// loads 4 groups of 16 elements (8 x 16 B in flight) before it casts, and a
// warp's loads and stores of one group cover contiguous 1 KB / 512 B.  The
// grid is the work (one CTA per 16384 elements), so CTAs come and go as
// the SMs free up instead of sweeping the tensor in lockstep.  Two tensors
// may share a launch (the X and W of a forward pass): CTAs [0, ctas0) take
// job 0, the rest job 1; the first CTA of a job also casts its last n % 16
// elements.
struct FlatJob {
    const uint4* x;
    int64_t n16;
    const uint16_t* xt;   // the last tail_n elements
    int tail_n;
    const float* scale;
    uint4* q;
    uint8_t* qtail;
    unsigned* amax_bits;
    ScaleUpd upd;   // upd.amax null: the scale is *scale
};

constexpr int kChunkGroups = 4 * kThreads;   // 16-element groups per CTA
// CTAs per tensor of the small-tensor cast: one cluster of 16 (a size
// beyond the portable 8, allowed per kernel; 6% less latency than 8 on a
// small layer's forward replayed from a CUDA graph)
constexpr int kSmallCtas = 16;
constexpr int kSmallThreads = 256;            // threads per CTA of the small-tensor cast

template <int FMT, bool AMAX, bool COUNT, bool UPD>
__global__ void __launch_bounds__(kThreads)
    quantize_chunk_kernel(FlatJob j0, FlatJob j1, int64_t ctas0, unsigned long long* counts) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const bool second = blockIdx.x >= ctas0;
    const FlatJob& j = second ? j1 : j0;
    const int64_t cta = second ? blockIdx.x - ctas0 : blockIdx.x;
    const float s = (UPD && j.upd.amax)
                        ? fused_dynamic_scale(j.upd, Fp8Traits<FMT>::max_finite,
                                              cta == 0 && threadIdx.x == 0)
                        : *j.scale;
    const SrSched key{};
    uint32_t m = 0;
    CastCounts cc;
    const int64_t g0 = cta * kChunkGroups + threadIdx.x;
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t g = g0 + u * kThreads;
        a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
        if (g < j.n16) {
            a[u] = ldg_stream(j.x + 2 * g);
            b[u] = ldg_stream(j.x + 2 * g + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t g = g0 + u * kThreads;
        if (g < j.n16) {
            if (AMAX) m = absmax_vec(absmax_vec(m, a[u]), b[u]);
            j.q[g] = cast16<FMT, COUNT, false>(a[u], b[u], s, cc, key, 0);
        }
    }
    if (cta == 0 && threadIdx.x < j.tail_n) {
        const uint32_t w = j.xt[threadIdx.x];
        if (AMAX) m = max(m, w & 0x7FFFu);
        const uint32_t code = COUNT ? cvt2c<FMT>(w & 0xFFFFu, s, cc) : cvt2<FMT>(w, s);
        j.qtail[threadIdx.x] = static_cast<uint8_t>(code & 0xFFu);
    }
    if (AMAX) cta_amax_commit(m, j.amax_bits);
    if (COUNT) cta_counts_commit(cc, counts);
}

// Dynamic scaling of small tensors (a small layer's X and W, or its dY):
// the amax, the scale computed from it and the cast in one launch, one
// cluster of kSmallCtas CTAs per tensor.  Each CTA reduces its share of the
// maximum; the cluster combines the CTAs' maxima through distributed shared
// memory; every thread derives the scale (the first thread of the cluster
// also writes the role's amax slot and state update) and the CTAs cast their
// shares.  This replaces the zeroing, amax and cast launches of the chunked
// path with the same maximum, the same scale function and the same
// conversion, so the codes and state are the same bits; the second read of
// the tensor comes from L2.  Job 1 may be empty (n16 = tail_n = 0).
template <int FMT>
__global__ void __cluster_dims__(kSmallCtas, 1, 1) __launch_bounds__(kSmallThreads)
    small_dynamic_cast_kernel(FlatJob j0, FlatJob j1, float* amax0, float* amax1) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ uint32_t warp_max[kSmallThreads / 32];
    __shared__ uint32_t cta_max;
    const bool second = static_cast<int>(blockIdx.x) >= kSmallCtas;
    const FlatJob& j = second ? j1 : j0;
    float* amax_slot = second ? amax1 : amax0;
    const int r = static_cast<int>(ptx::cluster_ctarank()), t = threadIdx.x;
    const int64_t stride = static_cast<int64_t>(kSmallCtas) * kSmallThreads;
    const int64_t g0 = static_cast<int64_t>(r) * kSmallThreads + t;
    uint32_t m2 = 0;
    for (int64_t g = g0; g < j.n16; g += stride)
        m2 = absmax_vec(absmax_vec(m2, ldg_stream(j.x + 2 * g)), ldg_stream(j.x + 2 * g + 1));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    if (r == 0 && t < j.tail_n) m = max(m, static_cast<uint32_t>(j.xt[t] & 0x7FFFu));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((t & 31) == 0) warp_max[t >> 5] = m;
    __syncthreads();
    if (t < 32) {
        uint32_t v = t < kSmallThreads / 32 ? warp_max[t] : 0u;
        v = __reduce_max_sync(0xFFFFFFFFu, v);
        if (t == 0) cta_max = v;
    }
    ptx::cluster_sync();   // every CTA's maximum is in its shared memory
    uint32_t bits = 0;
#pragma unroll
    for (int c = 0; c < kSmallCtas; ++c)
        bits = max(bits, ptx::ld_shared_cluster_u32(ptx::cluster_addr(&cta_max, c)));
    // the peers' reads of this CTA's maximum have been performed before it may
    // exit (release ordering: a load still in flight at a relaxed arrive could
    // reach a CTA that has already left)
    ptx::cluster_sync();
    const float a = __uint_as_float(bits << 16);
    const bool writer = r == 0 && t == 0;
    const float s = dynamic_scale_of(j.upd, Fp8Traits<FMT>::max_finite, a, writer);
    if (writer) *amax_slot = a;
    CastCounts cc;
    const SrSched key{};
    for (int64_t g = g0; g < j.n16; g += stride)
        j.q[g] = cast16<FMT, false, false>(ldg_stream(j.x + 2 * g), ldg_stream(j.x + 2 * g + 1), s,
                                           cc, key, 0);
    if (r == 0 && t < j.tail_n)
        j.qtail[t] = static_cast<uint8_t>(cvt2<FMT>(j.xt[t], s) & 0xFFu);
}

// Cast with fused transpose.  One CTA per 128 x 128 tile:
//  phase 1: each thread reads 16 consecutive bf16 of a row (2 x 16 B), writes
//           16 FP8 codes of q (16 B) and keeps them in shared memory;
//  phase 2: each thread gathers 4 x 4 byte blocks from shared memory,
//           transposes them with byte permutes and writes 4 codes to each of
//           4 rows of q_t (a warp covers 128 contiguous bytes per row).
// Shared-memory rows of 32 words are XOR-swizzled in groups of 4 words so
// that phase 1 stores stay 16-byte vectors and phase 2 reads spread over
// 8 banks.  rows and cols are multiples of 16.
__device__ __forceinline__ int tr_swz(int row) { return ((row >> 2) & 7) << 2; }

// Phase 2 of the transposing casts: the 128 x 128 tile of codes at (r0, c0),
// staged in S (rows of 32 words, swizzled by tr_swz), is written transposed
// to qt [cols x ld] (ld = row length of qt): each thread gathers 4 x 4 byte
// blocks, transposes them with byte permutes and writes 4 codes to each of 4
// rows of qt (a warp covers 128 contiguous bytes per row).
__device__ __forceinline__ void transpose_tile_out(const uint32_t* S, uint8_t* __restrict__ qt,
                                                   int64_t ld, int64_t r0, int64_t c0,
                                                   int64_t rows, int64_t cols) {
    const int t = threadIdx.x;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int b = it * kThreads + t;
        const int br = b & 31, bc = b >> 5;
        const int R = 4 * br;
        const uint32_t w0 = S[(R + 0) * 32 + (bc ^ tr_swz(R + 0))];
        const uint32_t w1 = S[(R + 1) * 32 + (bc ^ tr_swz(R + 1))];
        const uint32_t w2 = S[(R + 2) * 32 + (bc ^ tr_swz(R + 2))];
        const uint32_t w3 = S[(R + 3) * 32 + (bc ^ tr_swz(R + 3))];
        const uint32_t lo01 = __byte_perm(w0, w1, 0x5140), hi01 = __byte_perm(w0, w1, 0x7362);
        const uint32_t lo23 = __byte_perm(w2, w3, 0x5140), hi23 = __byte_perm(w2, w3, 0x7362);
        const uint32_t o[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                               __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
        const int64_t r = r0 + R, c = c0 + 4 * bc;
        if (r < rows) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (c + k < cols) *reinterpret_cast<uint32_t*>(qt + (c + k) * ld + r) = o[k];
        }
    }
}

// Column sums of one 128 x 128 bf16 tile for the bias gradient.  The tile
// is held as in the transposing cast: thread t has rows it*32 + t/8
// (it = 0..3) and columns 16*(t%8) .. +15 in va[it] (first 8) and vb[it]
// (last 8), zero outside the matrix.  Sums run over the thread's 4 rows,
// then over the 4 lanes of a warp that share the columns (xor 8, xor 16),
// then over the 8 warps in warp order, all in fp32 and in a fixed order, so
// the result does not depend on scheduling.  Threads 0..127 write column
// c0 + t of `prow` (one row of partial sums per 128-row tile).
// CTA-collective.
__device__ __forceinline__ void tile_column_sums(const uint4 (&va)[4], const uint4 (&vb)[4],
                                                 float* __restrict__ prow, int64_t cols,
                                                 int64_t c0) {
    __shared__ float red[kThreads / 32][128];
    float sum[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) sum[j] = 0.0f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const uint32_t w[8] = {va[it].x, va[it].y, va[it].z, va[it].w,
                               vb[it].x, vb[it].y, vb[it].z, vb[it].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sum[2 * e] = __fadd_rn(sum[2 * e], __uint_as_float(w[e] << 16));
            sum[2 * e + 1] = __fadd_rn(sum[2 * e + 1], __uint_as_float(w[e] & 0xFFFF0000u));
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        sum[j] = __fadd_rn(sum[j], __shfl_xor_sync(0xFFFFFFFFu, sum[j], 8));
        sum[j] = __fadd_rn(sum[j], __shfl_xor_sync(0xFFFFFFFFu, sum[j], 16));
    }
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 16; ++j) red[warp][lane * 16 + j] = sum[j];
    }
    __syncthreads();
    if (t < 128) {
        float v = red[0][t];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) v = __fadd_rn(v, red[w][t]);
        if (c0 + t < cols) prow[c0 + t] = v;
    }
}

// Round-to-nearest cast of the 128 x 128 tile at (r0, c0) of x [rows x
// cols] with its transposed copy, staged in S (128 rows of 32 words);
// optional fused amax, counters and bias-gradient sums.  CTA-collective.
template <int FMT, bool AMAX, bool COUNT, bool DBIAS>
__device__ __forceinline__ void rne_cast_transpose_tile(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t r0, int64_t c0, float s,
    uint8_t* __restrict__ q, uint8_t* __restrict__ qt, unsigned* amax_bits,
    unsigned long long* counts, float* __restrict__ dbias_partial, uint32_t* S) {
    CastCounts cc;
    const SrSched key{};
    const int t = threadIdx.x, cg = t & 7;
    uint32_t m = 0;
    // all of this thread's loads first (8 x 16 B in flight), then cast and store
    uint4 va[4], vb[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int64_t r = r0 + it * 32 + (t >> 3), c = c0 + cg * 16;
        va[it] = vb[it] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && c < cols) {
            const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
            va[it] = ldg_stream(src);
            vb[it] = ldg_stream(src + 1);
        }
    }
    if (DBIAS) tile_column_sums(va, vb, dbias_partial + (r0 >> 7) * cols, cols, c0);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rl = it * 32 + (t >> 3);
        const int64_t r = r0 + rl, c = c0 + cg * 16;
        const uint4 a = va[it], b = vb[it];
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && c < cols) {
            if (AMAX) m = absmax_vec(absmax_vec(m, a), b);
            out = cast16<FMT, COUNT, false>(a, b, s, cc, key, 0);
            *reinterpret_cast<uint4*>(q + r * cols + c) = out;
        }
        if (qt) *reinterpret_cast<uint4*>(&S[rl * 32 + ((cg * 4) ^ tr_swz(rl))]) = out;
    }
    if (qt) {   // (null: the bias-gradient sums without a transposed copy)
        __syncthreads();
        transpose_tile_out(S, qt, rows, r0, c0, rows, cols);
    }
    if (AMAX) cta_amax_commit(m, amax_bits);
    if (COUNT) cta_counts_commit(cc, counts);
}

template <int FMT, bool AMAX, bool COUNT, bool SR, bool DBIAS>
__global__ void __launch_bounds__(kThreads)
    quantize_transpose_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                              int64_t tiles_c, const float* __restrict__ scale_p,
                              uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
                              unsigned* amax_bits, unsigned long long* counts, SrKey sr_key,
                              float* __restrict__ dbias_partial,
                              const unsigned long long* key_dev) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    static_assert(!(SR && DBIAS), "the bias-gradient sums ride on the round-to-nearest cast");
    CastCounts cc;
    const SrSched key = sr_sched(sr_key_of(sr_key, SR ? key_dev : nullptr));
    __shared__ __align__(16) uint32_t S[128 * 32];
    const int64_t tile = blockIdx.x;
    const int64_t r0 = (tile / tiles_c) * 128, c0 = (tile % tiles_c) * 128;
    const float s = *scale_p;
    const int t = threadIdx.x;
    uint32_t m = 0;

    const int cg = t & 7;
    if constexpr (SR) {
        // stochastic rounding is ALU-heavy (one Philox call per 4 elements):
        // a rolled loop keeps the code small, and the arithmetic of one row
        // segment hides the latency of the next one's loads
#pragma unroll 1
        for (int it = 0; it < 4; ++it) {
            const int rl = it * 32 + (t >> 3);
            const int64_t r = r0 + rl, c = c0 + cg * 16;
            uint4 out = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows && c < cols) {
                const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
                const uint4 a = ldg_stream(src), b = ldg_stream(src + 1);
                if (AMAX) m = absmax_vec(absmax_vec(m, a), b);
                out = cast16<FMT, COUNT, SR>(a, b, s, cc, key, static_cast<uint64_t>(r * cols + c) >> 4);
                *reinterpret_cast<uint4*>(q + r * cols + c) = out;
            }
            *reinterpret_cast<uint4*>(&S[rl * 32 + ((cg * 4) ^ tr_swz(rl))]) = out;
        }
        __syncthreads();
        transpose_tile_out(S, qt, rows, r0, c0, rows, cols);
        if (AMAX) cta_amax_commit(m, amax_bits);
    } else {
        rne_cast_transpose_tile<FMT, AMAX, COUNT, DBIAS>(x, rows, cols, r0, c0, s, q, qt, amax_bits,
                                                         counts, dbias_partial, S);
    }
}

// One pass over the 128 x 128 tiles of two tensors (the X and W of a
// forward pass): tiles [0, tiles0) belong to job 0, the rest to job 1.  One
// launch instead of two, and the smaller tensor's tiles fill the other's
// last wave.
struct CastJob {
    const uint16_t* x;
    int64_t rows, cols, tiles_c;
    const float* scale;
    uint8_t* q;
    uint8_t* qt;
    unsigned* amax_bits;
};

template <int FMT, bool AMAX>
__global__ void __launch_bounds__(kThreads)
    quantize_transpose_pair_kernel(CastJob j0, CastJob j1, int64_t tiles0) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ __align__(16) uint32_t S[128 * 32];
    const bool second = blockIdx.x >= tiles0;
    const CastJob& j = second ? j1 : j0;
    const int64_t tile = second ? blockIdx.x - tiles0 : blockIdx.x;
    const int64_t r0 = (tile / j.tiles_c) * 128, c0 = (tile % j.tiles_c) * 128;
    rne_cast_transpose_tile<FMT, AMAX, false, false>(j.x, j.rows, j.cols, r0, c0, *j.scale, j.q,
                                                     j.qt, j.amax_bits, nullptr, nullptr, S);
}

// Bias-gradient partial sums without a cast (for the block-wise and per-row
// backward, whose dY casts have other layouts): one CTA per 128 x 128 tile
// of x [rows x cols] (cols % 16 == 0), the same loads and the same sums as
// the fused variant of the transposing cast.
__global__ void __launch_bounds__(kThreads)
    column_partial_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                          int64_t tiles_c, float* __restrict__ partial) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const int64_t tile = blockIdx.x;
    const int64_t r0 = (tile / tiles_c) * 128, c0 = (tile % tiles_c) * 128;
    const int t = threadIdx.x, cg = t & 7;
    uint4 va[4], vb[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int64_t r = r0 + it * 32 + (t >> 3), c = c0 + cg * 16;
        va[it] = vb[it] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && c < cols) {
            const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
            va[it] = ldg_stream(src);
            vb[it] = ldg_stream(src + 1);
        }
    }
    tile_column_sums(va, vb, partial + (r0 >> 7) * cols, cols, c0);
}

// dbias[n] = sum over the P partial rows of column n, in row order
// (+ the old dbias[n] when accumulating).
__global__ void dbias_finalize_kernel(const float* __restrict__ partial, int64_t P, int64_t cols,
                                      float* __restrict__ dbias, int accumulate) {
    // (tiny kernel: the next one may launch once the kernel before this one
    // has completed, not earlier, so a chain of launches cannot run ahead of
    // a large kernel)
    ptx::griddep_wait();   // the previous kernel's results are visible
    ptx::griddep_launch_dependents();
    const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (n >= cols) return;
    float v = 0.0f;
    for (int64_t p = 0; p < P; ++p) v = __fadd_rn(v, partial[p * cols + n]);
    dbias[n] = accumulate ? __fadd_rn(dbias[n], v) : v;
}

// The counter word of a device-held stochastic-rounding key moves on by
// one after a cast has used it.
__global__ void sr_advance_kernel(unsigned long long* key_dev) {
    // (tiny kernel: the next one may launch once the kernel before this one
    // has completed, not earlier, so a chain of launches cannot run ahead of
    // a large kernel)
    ptx::griddep_wait();   // the previous kernel's results are visible
    ptx::griddep_launch_dependents();
    key_dev[1] += 1ull;
}

// ----------------------------------------------------------- block casts

// 1x128: a half-warp per row segment (16 lanes x 8 elements); the segment's
// amax is a max-reduction over the 16 lanes.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
    quantize_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int pow2,
                          uint8_t* __restrict__ q, float* __restrict__ scale_inv) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    // a half-warp per 128-element segment, a warp per pair of segments; each
    // warp takes kU pairs per step with all their loads issued first, so that
    // enough bytes are in flight to cover the memory latency
    constexpr int kU = 4;
    const int64_t nseg = rows * (cols / 128);
    const int64_t npairs = (nseg + 1) / 2;
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t p0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         p0 < npairs; p0 += kU * warps) {
        uint4 v[kU];
        int64_t off[kU], seg[kU];
        bool valid[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t p = p0 + u * warps;
            seg[u] = 2 * p + (lane >> 4);
            valid[u] = p < npairs && seg[u] < nseg;
            // cols = 128 * KB: segment seg starts at element 128 * seg
            off[u] = seg[u] * 128 + sub * 8;
            v[u] = valid[u] ? ldg_stream(reinterpret_cast<const uint4*>(x + off[u]))
                            : make_uint4(0u, 0u, 0u, 0u);
        }
        // each half-warp's maxima of its kU segments; lane sub (< kU) of the
        // half computes the scale of segment sub and writes its factor, the
        // others take the scale by a shuffle (one division sequence per lane
        // instead of kU)
        uint32_t mu[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const uint32_t m2 = absmax_vec(0u, v[u]);
            uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            mu[u] = m;
        }
        uint32_t m_own = mu[0];
        int64_t seg_own = seg[0];
        bool valid_own = valid[0];
#pragma unroll
        for (int u = 1; u < kU; ++u)
            if (sub == u) {
                m_own = mu[u];
                seg_own = seg[u];
                valid_own = valid[u];
            }
        const float s_own = block_scale<FMT>(__uint_as_float(m_own << 16), pow2);
        if (sub < kU && valid_own) scale_inv[seg_own] = __fdiv_rn(1.0f, s_own);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const float s = __shfl_sync(0xFFFFFFFFu, s_own, (lane & 16) + u);
            if (valid[u])
                *reinterpret_cast<uint2*>(q + off[u]) =
                    make_uint2(cvt4<FMT>(v[u].x, v[u].y, s), cvt4<FMT>(v[u].z, v[u].w, s));
        }
    }
}

// 128x128: one CTA per tile; each thread holds 64 elements in registers
// while the CTA reduces the tile's amax.
// With qt (nullable): also the transposed codes q_t [C x R] -- the same
// codes, since a 128 x 128 block keeps its scale under transposition -- and
// the transposed scale array scale_inv_t [C/128][R/128].
template <int FMT>
__global__ void __launch_bounds__(kThreads)
    quantize_128x128_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int pow2,
                            uint8_t* __restrict__ q, float* __restrict__ scale_inv,
                            uint8_t* __restrict__ qt, float* __restrict__ scale_inv_t) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ uint32_t warp_max[kThreads / 32];
    __shared__ __align__(16) uint32_t S[128 * 32];
    const int64_t KB = cols / 128;
    const int64_t br = blockIdx.x / KB, bc = blockIdx.x % KB;
    const int t = threadIdx.x;
    uint4 v[8];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = br * 128 + i * 16 + (t >> 4), c = bc * 128 + (t & 15) * 8;
        v[i] = ldg_stream(reinterpret_cast<const uint4*>(x + r * cols + c));
        m2 = absmax_vec(m2, v[i]);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((t & 31) == 0) warp_max[t >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, warp_max[w]);
    const float s = block_scale<FMT>(__uint_as_float(m << 16), pow2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rl = i * 16 + (t >> 4);
        const int64_t r = br * 128 + rl, c = bc * 128 + (t & 15) * 8;
        const uint2 codes = make_uint2(cvt4<FMT>(v[i].x, v[i].y, s), cvt4<FMT>(v[i].z, v[i].w, s));
        *reinterpret_cast<uint2*>(q + r * cols + c) = codes;
        if (qt) *reinterpret_cast<uint2*>(&S[rl * 32 + (((t & 15) * 2) ^ tr_swz(rl))]) = codes;
    }
    if (t == 0) scale_inv[br * KB + bc] = __fdiv_rn(1.0f, s);
    if (qt) {
        __syncthreads();
        transpose_tile_out(S, qt, rows, br * 128, bc * 128, rows, cols);
        if (t == 0) scale_inv_t[bc * (rows / 128) + br] = __fdiv_rn(1.0f, s);
    }
}

// Dual 1x128 cast for the block-wise backward: one read of each 128 x 128
// bf16 tile gives
//   q   [R x C]  with one scale per 1x128 row segment   (scale_inv [R][C/128])
//   q_t [C x R]  with one scale per 1x128 segment of a column of x, i.e. the
//                1x128 block cast of x^T                  (scale_inv_t [C][R/128]).
// R and C are multiples of 128.
//
// Persistent CTAs (two per SM) walk the tiles; each keeps kDualStages tiles in
// flight in a ring of shared-memory stages filled by TMA, so that the next
// tile arrives while the current one is reduced and written (one CTA per tile
// and plain loads left each tile's load latency exposed: about 0.65 of the
// HBM bandwidth).  Per tile, thread t holds rows it*32 + t/8 (it = 0..3) and
// columns 16*(t%8) .. +15:
//   rows     the 8 threads of a row reduce its 128-element amax with shuffles,
//            cast and write q (16 bytes each) and the row's scale;
//   columns  the column maxima are reduced from registers (4 rows per thread,
//            4 lanes per warp, then the 8 warps through shared memory); each
//            thread casts its elements with their columns' scales into the
//            byte staging S, which transpose_tile_out writes to q_t in whole
//            128-byte row segments.
constexpr int kDualStages = 2;
constexpr int kDualTileBytes = 128 * 128 * 2;
constexpr int kDualSmem = kDualStages * kDualTileBytes + 64 + 1024;

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_1x128_dual_kernel(const __grid_constant__ CUtensorMap tmX, int64_t rows, int64_t cols,
                               int64_t tiles_c, int64_t tiles, int pow2, uint8_t* __restrict__ q,
                               float* __restrict__ scale_inv, uint8_t* __restrict__ qt,
                               float* __restrict__ scale_inv_t, unsigned* status) {
    ptx::griddep_launch_dependents();
    __shared__ __align__(16) uint32_t S[128 * 32];          // column-scaled codes, swizzled rows
    __shared__ uint32_t colpart[kThreads / 32][64];         // per warp: 128 column maxima, 2 per word
    __shared__ __align__(16) float colscale[128];
    __shared__ uint32_t abort_word;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kDualStages * kDualTileBytes);
    const int t = threadIdx.x, cg = t & 7;
    if (t == 0) {
        for (int st = 0; st < kDualStages; ++st) ptx::mbar_init(&full[st], 1);
        abort_word = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    ptx::griddep_wait();   // the previous kernel's results are visible
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < tiles ? (tiles - first + step - 1) / step : 0;
    // the k-th tile of this CTA goes to stage k % kDualStages
    auto issue = [&](int64_t k) {
        const int64_t tile = first + k * step;
        const int st = static_cast<int>(k % kDualStages);
        ptx::mbar_arrive_expect_tx(&full[st], kDualTileBytes);
        ptx::tma_load_2d(ring + st * kDualTileBytes, &tmX, &full[st],
                         static_cast<int32_t>((tile % tiles_c) * 128),
                         static_cast<int32_t>((tile / tiles_c) * 128));
    };
    if (t == 0)
        for (int64_t k = 0; k < mine && k < kDualStages; ++k) issue(k);
    int64_t k = 0;
    for (; k < mine; ++k) {
        const int st = static_cast<int>(k % kDualStages);
        const uint32_t par = static_cast<uint32_t>(k / kDualStages) & 1u;
        const int64_t tile = first + k * step;
        const int64_t r0 = (tile / tiles_c) * 128, c0 = (tile % tiles_c) * 128;
        // every thread sees the stage's bytes land; the verdict is the CTA's
        // (all threads leave together if a wait gave up)
        const bool ok = ptx::mbar_wait(&full[st], par, &abort_word);
        if (!__syncthreads_and(ok)) break;
        const uint8_t* tile_s = ring + st * kDualTileBytes;
        uint4 va[4], vb[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const uint4* src = reinterpret_cast<const uint4*>(tile_s + (it * 32 + (t >> 3)) * 256 + cg * 32);
            va[it] = src[0];
            vb[it] = src[1];
        }
        __syncthreads();   // the stage has been read: refill it with tile k + kDualStages
        if (t == 0 && k + kDualStages < mine) issue(k + kDualStages);
        // column maxima from registers: this thread's 4 rows of its 16 columns,
        // then the 4 lanes of the warp with the same columns, then the 8 warps
        uint32_t cm[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            cm[0] = absmax2(cm[0], va[it].x); cm[1] = absmax2(cm[1], va[it].y);
            cm[2] = absmax2(cm[2], va[it].z); cm[3] = absmax2(cm[3], va[it].w);
            cm[4] = absmax2(cm[4], vb[it].x); cm[5] = absmax2(cm[5], vb[it].y);
            cm[6] = absmax2(cm[6], vb[it].z); cm[7] = absmax2(cm[7], vb[it].w);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            cm[j] = __vmaxu2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 8));
            cm[j] = __vmaxu2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 16));
        }
        if ((t & 31) < 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) colpart[t >> 5][cg * 8 + j] = cm[j];
        }
        // row blocks: each 128-element row segment of the tile has its own scale.
        // The 8 threads of a row reduce the amaxes of their 4 rows; then lane
        // cg = it of each row group computes the scale of row `it` (one
        // division sequence per warp instead of four) and the others take it
        // by a shuffle
        uint32_t mrow[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const uint32_t m2 = absmax_vec(absmax_vec(0u, va[it]), vb[it]);
            uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            mrow[it] = m;
        }
        const uint32_t m_own = cg == 0 ? mrow[0] : cg == 1 ? mrow[1] : cg == 2 ? mrow[2] : mrow[3];
        const float sc_own = block_scale<FMT>(__uint_as_float(m_own << 16), pow2);
        if (cg < 4)
            scale_inv[(r0 + cg * 32 + (t >> 3)) * (cols / 128) + c0 / 128] = __fdiv_rn(1.0f, sc_own);
        const int group = (t & 31) & ~7;   // first lane of this thread's row group
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const uint4 a = va[it], b = vb[it];
            const float sc = __shfl_sync(0xFFFFFFFFu, sc_own, group + it);
            const int64_t r = r0 + it * 32 + (t >> 3);
            *reinterpret_cast<uint4*>(q + r * cols + c0 + cg * 16) =
                make_uint4(cvt4<FMT>(a.x, a.y, sc), cvt4<FMT>(a.z, a.w, sc), cvt4<FMT>(b.x, b.y, sc),
                           cvt4<FMT>(b.z, b.w, sc));
        }
        __syncthreads();
        // column blocks: one scale per column of the tile (thread c < 128)
        if (t < 128) {
            uint32_t w2 = 0;
#pragma unroll
            for (int g = 0; g < kThreads / 32; ++g) w2 = __vmaxu2(w2, colpart[g][t >> 1]);
            const uint32_t m = (t & 1) ? (w2 >> 16) : (w2 & 0xFFFFu);
            const float sc = block_scale<FMT>(__uint_as_float(m << 16), pow2);
            colscale[t] = sc;
            scale_inv_t[(c0 + t) * (rows / 128) + r0 / 128] = __fdiv_rn(1.0f, sc);
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int rl = it * 32 + (t >> 3);
            const uint32_t in[8] = {va[it].x, va[it].y, va[it].z, va[it].w,
                                    vb[it].x, vb[it].y, vb[it].z, vb[it].w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 cs = *reinterpret_cast<const float4*>(&colscale[cg * 16 + 4 * j]);
                const uint32_t w0 = in[2 * j], w1 = in[2 * j + 1];
                const float f0 = __fmul_rn(__uint_as_float(w0 << 16), cs.x);
                const float f1 = __fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), cs.y);
                const float f2 = __fmul_rn(__uint_as_float(w1 << 16), cs.z);
                const float f3 = __fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), cs.w);
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f0, f1), __NV_SATFINITE, Fp8Traits<FMT>::kind);
                const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f2, f3), __NV_SATFINITE, Fp8Traits<FMT>::kind);
                o[j] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(&S[rl * 32 + ((cg * 4) ^ tr_swz(rl))]) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
        transpose_tile_out(S, qt, rows, r0, c0, rows, cols);
        __syncthreads();   // S, colpart and colscale are free for the next tile
    }
    if (t == 0) {
        if (k < mine) {
            // a wait gave up: let the copies already issued into the ring land
            // (bounded) before the CTA's shared memory is released
            uint32_t never = 0;
            for (int64_t j = k; j < mine && j < k + kDualStages; ++j)
                ptx::mbar_wait(&full[j % kDualStages],
                               static_cast<uint32_t>(j / kDualStages) & 1u, &never);
            if (status) atomicOr(status, 1u);   // bit 0: a bounded wait gave up
        }
    }
}

// ------------------------------------------------------ per-row scaling

// Per-row cast: one CTA per row, the row's amax (pass 1), then the cast with
// the row's scale (pass 2, the re-read hits L2).  scale_inv[row] = 1/s.
// cols is a multiple of 8.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
    quantize_row_kernel(const uint16_t* __restrict__ x, int64_t cols, int pow2,
                        uint8_t* __restrict__ q, float* __restrict__ scale_inv) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ uint32_t warp_max[kThreads / 32];
    const int64_t row = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(x + row * cols);
    const int64_t nv = cols / 8;
    uint32_t m2 = 0;
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) m2 = absmax_vec(m2, src[i]);
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, warp_max[w]);
    const float s = block_scale<FMT>(__uint_as_float(m << 16), pow2);
    uint2* dst = reinterpret_cast<uint2*>(q + row * cols);
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
        const uint4 v = src[i];
        dst[i] = make_uint2(cvt4<FMT>(v.x, v.y, s), cvt4<FMT>(v.z, v.w, s));
    }
    if (threadIdx.x == 0) scale_inv[row] = __fdiv_rn(1.0f, s);
}

// The per-row cast together with the per-row cast of x^T (one scale per row
// and one per column) in two reads of x.  Pass 1: each CTA takes `group`
// 128 x 128 tiles down one column of tiles and raises the row maxima
// rowmax[r] (one atomicMax per row and tile) and the column maxima colmax[c]
// (one atomicMax per column for the group, from maxima kept in registers
// across it) -- fp32 bit patterns of |bf16| maxima, in arrays zeroed
// beforehand.  Groups of 4 take 3-4% off the large shapes (a quarter of the
// column atomics); small shapes keep groups of 1, which fill the GPU.  rows,
// cols: multiples of 16.

__global__ void __launch_bounds__(kThreads)
    row_col_amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                        int64_t tiles_c, int group, unsigned* __restrict__ rowmax,
                        unsigned* __restrict__ colmax) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ uint32_t colpart[kThreads / 32][64];
    const int64_t c0 = (blockIdx.x % tiles_c) * 128;
    const int64_t rg0 = (blockIdx.x / tiles_c) * (128 * static_cast<int64_t>(group));
    const int t = threadIdx.x, cg = t & 7;
    uint32_t cm[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int k = 0; k < group; ++k) {
        const int64_t r0 = rg0 + k * 128;
        if (r0 >= rows) break;
        uint4 va[4], vb[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int64_t r = r0 + it * 32 + (t >> 3), c = c0 + cg * 16;
            va[it] = vb[it] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows && c < cols) {
                const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
                va[it] = ldg_stream(src);
                vb[it] = ldg_stream(src + 1);
            }
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const uint4 a = va[it], b = vb[it];
            cm[0] = absmax2(cm[0], a.x); cm[1] = absmax2(cm[1], a.y);
            cm[2] = absmax2(cm[2], a.z); cm[3] = absmax2(cm[3], a.w);
            cm[4] = absmax2(cm[4], b.x); cm[5] = absmax2(cm[5], b.y);
            cm[6] = absmax2(cm[6], b.z); cm[7] = absmax2(cm[7], b.w);
            // the row's maximum over the tile: the 8 lanes that hold the row
            const uint32_t m2 = absmax_vec(absmax_vec(0u, a), b);
            uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            const int64_t r = r0 + it * 32 + (t >> 3);
            if (cg == 0 && m && r < rows) atomicMax(&rowmax[r], m << 16);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        cm[j] = __vmaxu2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 8));
        cm[j] = __vmaxu2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 16));
    }
    if ((t & 31) < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) colpart[t >> 5][cg * 8 + j] = cm[j];
    }
    __syncthreads();
    if (t < 128 && c0 + t < cols) {
        uint32_t w2 = 0;
#pragma unroll
        for (int g = 0; g < kThreads / 32; ++g) w2 = __vmaxu2(w2, colpart[g][t >> 1]);
        const uint32_t m = (t & 1) ? (w2 >> 16) : (w2 & 0xFFFFu);
        if (m) atomicMax(&colmax[c0 + t], m << 16);
    }
}

// Pass 2: each tile cast twice from registers -- with its rows' scales into
// q, with its columns' scales into the byte staging that the per-tensor
// transpose writes out as q_t.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
    quantize_row_col_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                            int64_t tiles_c, int pow2, const unsigned* __restrict__ rowmax,
                            const unsigned* __restrict__ colmax, uint8_t* __restrict__ q,
                            uint8_t* __restrict__ qt) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // the previous kernel's results are visible
    __shared__ __align__(16) uint32_t S[128 * 32];
    __shared__ __align__(16) float colscale[128];
    const int64_t tile = blockIdx.x;
    const int64_t r0 = (tile / tiles_c) * 128, c0 = (tile % tiles_c) * 128;
    const int t = threadIdx.x, cg = t & 7;
    if (t < 128)
        colscale[t] = c0 + t < cols ? block_scale<FMT>(__uint_as_float(colmax[c0 + t]), pow2) : 1.0f;
    uint4 va[4], vb[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int64_t r = r0 + it * 32 + (t >> 3), c = c0 + cg * 16;
        va[it] = vb[it] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && c < cols) {
            const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + c);
            va[it] = ldg_stream(src);
            vb[it] = ldg_stream(src + 1);
        }
    }
    // the rows' scales: lane cg (< 4) of each row group computes the scale of
    // the group's row in iteration cg (one division sequence per thread
    // instead of four) and the others take it by a shuffle
    const int64_t r_own = r0 + (cg & 3) * 32 + (t >> 3);
    const float sc_own =
        block_scale<FMT>(__uint_as_float(r_own < rows ? rowmax[r_own] : 0u), pow2);
    const int group = (t & 31) & ~7;   // first lane of this thread's row group
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rl = it * 32 + (t >> 3);
        const int64_t r = r0 + rl, c = c0 + cg * 16;
        const uint4 a = va[it], b = vb[it];
        const float rs = __shfl_sync(0xFFFFFFFFu, sc_own, group + it);
        if (r < rows && c < cols) {
            *reinterpret_cast<uint4*>(q + r * cols + c) =
                make_uint4(cvt4<FMT>(a.x, a.y, rs), cvt4<FMT>(a.z, a.w, rs),
                           cvt4<FMT>(b.x, b.y, rs), cvt4<FMT>(b.z, b.w, rs));
        }
        const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 cs = *reinterpret_cast<const float4*>(&colscale[cg * 16 + 4 * k]);
            const uint32_t w0 = in[2 * k], w1 = in[2 * k + 1];
            const float f0 = __fmul_rn(__uint_as_float(w0 << 16), cs.x);
            const float f1 = __fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), cs.y);
            const float f2 = __fmul_rn(__uint_as_float(w1 << 16), cs.z);
            const float f3 = __fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), cs.w);
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f0, f1), __NV_SATFINITE, Fp8Traits<FMT>::kind);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f2, f3), __NV_SATFINITE, Fp8Traits<FMT>::kind);
            o[k] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(&S[rl * 32 + ((cg * 4) ^ tr_swz(rl))]) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
    transpose_tile_out(S, qt, rows, r0, c0, rows, cols);
}

// a[i] = 1 / s(amax_i) for i < na, then b[i] likewise for i < nb, in place
// over the row and column amaxes: one launch for both.
template <int FMT>
__global__ void row_col_scale_finalize_kernel(float* __restrict__ a, int64_t na,
                                              float* __restrict__ b, int64_t nb, int pow2) {
    // (tiny kernel: the next one may launch once the kernel before this one
    // has completed, not earlier, so a chain of launches cannot run ahead of
    // a large kernel)
    ptx::griddep_wait();   // the previous kernel's results are visible
    ptx::griddep_launch_dependents();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    float* p = i < na ? a + i : (i - na < nb ? b + (i - na) : nullptr);
    if (p) *p = __fdiv_rn(1.0f, block_scale<FMT>(*p, pow2));
}

int grid_for(int64_t work_items, int per_cta) {
    const int64_t need = (work_items + per_cta - 1) / per_cta;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

// a[0..na) = 0 and b[0..nb) = 0 (b nullable): the maxima that the casts
// raise atomically start from zero.  A kernel rather than a memset, so that it
// takes part in programmatic dependent launch like the kernels around it.
__global__ void zero_words_kernel(float* __restrict__ a, int64_t na, float* __restrict__ b,
                                  int64_t nb) {
    // (tiny kernel: the next one may launch once the kernel before this one
    // has completed, not earlier, so a chain of launches cannot run ahead of
    // a large kernel)
    ptx::griddep_wait();   // the previous kernel's results are visible
    ptx::griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb;
         i += stride) {
        if (i < na) a[i] = 0.0f;
        else b[i - na] = 0.0f;
    }
}

cudaError_t launch_zero(float* a, int64_t na, float* b, int64_t nb, cudaStream_t stream) {
    const int64_t n = na + (b ? nb : 0);
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    launch_pdl(zero_words_kernel, dim3(static_cast<unsigned>(blocks < 1024 ? blocks : 1024)),
               dim3(256), 0, stream, a, na, b, b ? nb : int64_t{0});
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_amax_pair(const void* x0, int64_t n0, float* amax0, const void* x1, int64_t n1,
                             float* amax1, cudaStream_t stream) {
    cudaError_t e = launch_zero(amax0, 1, amax1, 1, stream);
    if (e != cudaSuccess || n0 + n1 == 0) return e;
    auto job = [](const void* x, int64_t n, float* amax) {
        const int64_t nvec = n / 8;
        return AmaxJob{static_cast<const uint4*>(x), nvec,
                       static_cast<const uint16_t*>(x) + nvec * 8, static_cast<int>(n - nvec * 8),
                       reinterpret_cast<unsigned*>(amax)};
    };
    const AmaxJob j0 = job(x0, n0, amax0), j1 = job(x1, n1, amax1);
    const int c0 = n0 ? grid_for(j0.nvec + 1, kThreads * 4) : 0;
    const int c1 = n1 ? grid_for(j1.nvec + 1, kThreads * 4) : 0;
    launch_pdl(amax_kernel, dim3(static_cast<unsigned>(c0 + c1)), dim3(kThreads), 0, stream, j0, j1, c0);
    return cudaGetLastError();
}

cudaError_t launch_amax(const void* x, int64_t n, float* amax, cudaStream_t stream) {
    return launch_amax_pair(x, n, amax, nullptr, 0, nullptr, stream);
}

cudaError_t launch_update_scale(const float* amax, float* history, int32_t* pos, int H, int algo,
                                int fmt, int margin, int pow2, float* scale, float* scale_inv,
                                int nroles, cudaStream_t stream, float* saved, int save_after) {
    const float fmax = fmt == 0 ? 448.0f : 57344.0f;
    launch_pdl(update_scale_kernel, dim3(nroles), dim3(32), 0, stream, amax, history, pos, H, algo, fmax, margin,
                                                   pow2, scale, scale_inv, saved, save_after,
                                                   device_status_word());
    return cudaGetLastError();
}

FlatJob flat_job(const void* x, int64_t n, const float* scale, uint8_t* q, float* amax) {
    const int64_t n16 = n / 16;
    return FlatJob{static_cast<const uint4*>(x), n16, static_cast<const uint16_t*>(x) + n16 * 16,
                   static_cast<int>(n - n16 * 16), scale, reinterpret_cast<uint4*>(q), q + n16 * 16,
                   reinterpret_cast<unsigned*>(amax), ScaleUpd{}};
}

int64_t chunk_ctas(const FlatJob& j) {
    // a job without elements still takes one CTA when it carries a fused
    // update, so that its state is written
    if (j.n16 == 0 && j.tail_n == 0) return j.upd.amax ? 1 : 0;
    const int64_t c = (j.n16 + kChunkGroups - 1) / kChunkGroups;
    return c < 1 ? 1 : c;
}

template <int FMT, bool AMAX, bool COUNT, bool UPD = false>
static void launch_chunk(const FlatJob& j0, const FlatJob& j1, unsigned long long* counts,
                         cudaStream_t stream) {
    const int64_t c0 = chunk_ctas(j0), c1 = chunk_ctas(j1);
    if (c0 + c1 == 0) return;
    launch_pdl(quantize_chunk_kernel<FMT, AMAX, COUNT, UPD>, dim3(static_cast<unsigned>(c0 + c1)),
               dim3(kThreads), 0, stream, j0, j1, c0, counts);
}

template <int FMT, bool AMAX, bool COUNT, bool SR>
static void launch_flat(const void* x, int64_t n, const float* scale, uint8_t* q, float* amax,
                        unsigned long long* counts, const SrKey& key, cudaStream_t stream,
                        const unsigned long long* key_dev = nullptr) {
    if constexpr (!SR) {   // round to nearest: one chunk per CTA
        launch_chunk<FMT, AMAX, COUNT>(flat_job(x, n, scale, q, amax), FlatJob{}, counts, stream);
    } else {               // stochastic rounding: grid-stride, bound by integer issue
        const int64_t n16 = n / 16;
        const int tail_n = static_cast<int>(n - n16 * 16);
        launch_pdl(quantize_flat_kernel<FMT, AMAX, COUNT, SR>, dim3(grid_for(n16 + 1, kThreads * 2)),
                   dim3(kThreads), 0, stream, static_cast<const uint4*>(x), n16,
                   static_cast<const uint16_t*>(x) + n16 * 16, tail_n, scale,
                   reinterpret_cast<uint4*>(q), q + n16 * 16, reinterpret_cast<unsigned*>(amax),
                   counts, key, key_dev);
    }
}

template <int FMT, bool AMAX, bool COUNT, bool SR, bool DBIAS = false>
static void launch_transpose(const void* x, int64_t rows, int64_t cols, const float* scale,
                             uint8_t* q, uint8_t* qt, float* amax, unsigned long long* counts,
                             const SrKey& key, cudaStream_t stream, float* dbias_partial = nullptr,
                             const unsigned long long* key_dev = nullptr) {
    const int64_t tiles_c = (cols + 127) / 128, tiles_r = (rows + 127) / 128;
    launch_pdl(quantize_transpose_kernel<FMT, AMAX, COUNT, SR, DBIAS>, dim3(static_cast<unsigned>(tiles_r * tiles_c)), dim3(kThreads), 0, stream, 
        static_cast<const uint16_t*>(x), rows, cols, tiles_c, scale, q, qt,
        reinterpret_cast<unsigned*>(amax), counts, key, dbias_partial, key_dev);
}

template <int FMT, bool AMAX, bool SR>
static void launch_cast(const void* x, int64_t rows, int64_t cols, const float* scale, uint8_t* q,
                        uint8_t* q_t, float* amax, unsigned long long* counts, const SrKey& key,
                        cudaStream_t stream, float* dbias_partial,
                        const unsigned long long* key_dev) {
    if constexpr (!SR) {
        if (dbias_partial) {   // the bias-gradient sums ride on the tiled cast (q_t nullable)
            launch_transpose<FMT, AMAX, false, false, true>(x, rows, cols, scale, q, q_t, amax,
                                                            nullptr, key, stream, dbias_partial);
            return;
        }
    }
    if constexpr (SR) {
        if (q_t) launch_transpose<FMT, AMAX, false, true>(x, rows, cols, scale, q, q_t, amax, nullptr, key, stream, nullptr, key_dev);
        else launch_flat<FMT, AMAX, false, true>(x, rows * cols, scale, q, amax, nullptr, key, stream, key_dev);
    } else if (q_t) {
        if (counts) launch_transpose<FMT, AMAX, true, false>(x, rows, cols, scale, q, q_t, amax, counts, key, stream);
        else launch_transpose<FMT, AMAX, false, false>(x, rows, cols, scale, q, q_t, amax, counts, key, stream);
    } else {
        if (counts) launch_flat<FMT, AMAX, true, false>(x, rows * cols, scale, q, amax, counts, key, stream);
        else launch_flat<FMT, AMAX, false, false>(x, rows * cols, scale, q, amax, counts, key, stream);
    }
}

template <bool SR>
static cudaError_t quantize_tensor(const void* x, int64_t rows, int64_t cols, int fmt,
                                   const float* scale, uint8_t* q, uint8_t* q_t, float* amax,
                                   unsigned long long* counts, const SrKey& key,
                                   cudaStream_t stream, float* dbias_partial = nullptr,
                                   const unsigned long long* key_dev = nullptr) {
    const int64_t n = rows * cols;
    if (amax) {
        cudaError_t e = launch_zero(amax, 1, nullptr, 0, stream);
        if (e != cudaSuccess) return e;
    }
    if (n == 0) return cudaSuccess;
    const bool A = amax != nullptr;
    if (fmt == 0) {
        if (A) launch_cast<0, true, SR>(x, rows, cols, scale, q, q_t, amax, counts, key, stream, dbias_partial, key_dev);
        else launch_cast<0, false, SR>(x, rows, cols, scale, q, q_t, amax, counts, key, stream, dbias_partial, key_dev);
    } else {
        if (A) launch_cast<1, true, SR>(x, rows, cols, scale, q, q_t, amax, counts, key, stream, dbias_partial, key_dev);
        else launch_cast<1, false, SR>(x, rows, cols, scale, q, q_t, amax, counts, key, stream, dbias_partial, key_dev);
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_tensor(const void* x, int64_t rows, int64_t cols, int fmt,
                                   const float* scale, uint8_t* q, uint8_t* q_t, float* amax,
                                   cudaStream_t stream, unsigned long long* counts,
                                   float* dbias_partial) {
    return quantize_tensor<false>(x, rows, cols, fmt, scale, q, q_t, amax, counts, SrKey{},
                                  stream, dbias_partial);
}

cudaError_t launch_small_dynamic_cast(const void* x0, int64_t n0, uint8_t* q0, float* amax0,
                                      const ScaleUpd& upd0, const void* x1, int64_t n1,
                                      uint8_t* q1, float* amax1, const ScaleUpd* upd1, int fmt,
                                      cudaStream_t stream) {
    if (n0 > kSmallDynamicElems || n1 > kSmallDynamicElems || (n1 && !upd1))
        return cudaErrorInvalidValue;
    FlatJob f0 = flat_job(x0, n0, nullptr, q0, nullptr);
    FlatJob f1 = flat_job(x1, n1, nullptr, q1, nullptr);
    f0.upd = upd0;
    if (upd1) f1.upd = *upd1;
    const unsigned grid = static_cast<unsigned>(kSmallCtas * (upd1 ? 2 : 1));
    {
        // clusters beyond 8 CTAs are allowed per kernel, once per device
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
        const bool cached = dev >= 0 && dev < 64;
        std::lock_guard<std::mutex> lock(mu);
        if (!cached || !done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(small_dynamic_cast_kernel<0>,
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(small_dynamic_cast_kernel<1>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            if (cached) done[dev] = true;
        }
    }
    if (fmt == 0)
        launch_pdl(small_dynamic_cast_kernel<0>, dim3(grid), dim3(kSmallThreads), 0, stream, f0, f1,
                   amax0, amax1);
    else
        launch_pdl(small_dynamic_cast_kernel<1>, dim3(grid), dim3(kSmallThreads), 0, stream, f0, f1,
                   amax0, amax1);
    return cudaGetLastError();
}

cudaError_t launch_quantize_pair(const void* x0, int64_t rows0, int64_t cols0, const float* scale0,
                                 uint8_t* q0, uint8_t* qt0, float* amax0, const void* x1,
                                 int64_t rows1, int64_t cols1, const float* scale1, uint8_t* q1,
                                 uint8_t* qt1, float* amax1, int fmt, cudaStream_t stream,
                                 const ScaleUpd* upd0, const ScaleUpd* upd1) {
    // a fused update rides on the chunked cast without a fused amax only
    if ((upd0 || upd1) && (qt0 || qt1 || amax0)) return cudaErrorInvalidValue;
    const bool A = amax0 != nullptr;
    if (A) {
        const cudaError_t e = launch_zero(amax0, 1, amax1, 1, stream);
        if (e != cudaSuccess) return e;
    }
    auto job = [](const void* x, int64_t rows, int64_t cols, const float* scale, uint8_t* q,
                  uint8_t* qt, float* amax) {
        return CastJob{static_cast<const uint16_t*>(x), rows, cols, (cols + 127) / 128, scale, q,
                       qt, reinterpret_cast<unsigned*>(amax)};
    };
    if (!qt0 && !qt1) {   // no transposed copies: one chunked cast over both tensors
        FlatJob f0 = flat_job(x0, rows0 * cols0, scale0, q0, amax0);
        FlatJob f1 = flat_job(x1, rows1 * cols1, scale1, q1, amax1);
        if (upd0) f0.upd = *upd0;
        if (upd1) f1.upd = *upd1;
        const bool U = upd0 || upd1;
        if (fmt == 0) {
            if (A) launch_chunk<0, true, false>(f0, f1, nullptr, stream);
            else if (U) launch_chunk<0, false, false, true>(f0, f1, nullptr, stream);
            else launch_chunk<0, false, false>(f0, f1, nullptr, stream);
        } else {
            if (A) launch_chunk<1, true, false>(f0, f1, nullptr, stream);
            else if (U) launch_chunk<1, false, false, true>(f0, f1, nullptr, stream);
            else launch_chunk<1, false, false>(f0, f1, nullptr, stream);
        }
        return cudaGetLastError();
    }
    const CastJob j0 = job(x0, rows0, cols0, scale0, q0, qt0, amax0);
    const CastJob j1 = job(x1, rows1, cols1, scale1, q1, qt1, amax1);
    const int64_t t0 = rows0 * cols0 ? ((rows0 + 127) / 128) * j0.tiles_c : 0;
    const int64_t t1 = rows1 * cols1 ? ((rows1 + 127) / 128) * j1.tiles_c : 0;
    if (t0 + t1 == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(t0 + t1);
    if (fmt == 0) {
        if (A) launch_pdl(quantize_transpose_pair_kernel<0, true>, dim3(grid), dim3(kThreads), 0, stream, j0, j1, t0);
        else launch_pdl(quantize_transpose_pair_kernel<0, false>, dim3(grid), dim3(kThreads), 0, stream, j0, j1, t0);
    } else {
        if (A) launch_pdl(quantize_transpose_pair_kernel<1, true>, dim3(grid), dim3(kThreads), 0, stream, j0, j1, t0);
        else launch_pdl(quantize_transpose_pair_kernel<1, false>, dim3(grid), dim3(kThreads), 0, stream, j0, j1, t0);
    }
    return cudaGetLastError();
}

cudaError_t launch_dbias(const void* x, int64_t rows, int64_t cols, float* partial,
                         bool partial_ready, float* dbias, int accumulate, cudaStream_t stream) {
    if (cols == 0) return cudaSuccess;
    const int64_t P = (rows + 127) / 128;
    if (!partial_ready && rows > 0) {
        const int64_t tiles_c = (cols + 127) / 128;
        launch_pdl(column_partial_kernel, dim3(static_cast<unsigned>(P * tiles_c)), dim3(kThreads), 0, stream, 
            static_cast<const uint16_t*>(x), rows, cols, tiles_c, partial);
    }
    launch_pdl(dbias_finalize_kernel, dim3(static_cast<unsigned>((cols + 255) / 256)), dim3(256), 0, stream, 
        partial, P, cols, dbias, accumulate);
    return cudaGetLastError();
}

cudaError_t launch_quantize_sr(const void* x, int64_t rows, int64_t cols, int fmt,
                               const float* scale, uint64_t seed, uint64_t offset, uint8_t* q,
                               uint8_t* q_t, float* amax, cudaStream_t stream,
                               uint64_t* key_dev) {
    const SrKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32),
                    static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32)};
    auto* kd = reinterpret_cast<unsigned long long*>(key_dev);
    cudaError_t e = quantize_tensor<true>(x, rows, cols, fmt, scale, q, q_t, amax, nullptr, key,
                                          stream, nullptr, kd);
    if (e != cudaSuccess || !key_dev) return e;
    launch_pdl(sr_advance_kernel, dim3(1), dim3(1), 0, stream, kd);
    return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_row(const uint16_t* xs, int64_t rows, int64_t cols, int pow2, uint8_t* q,
                              float* scale_inv, uint8_t* q_t, float* scale_inv_t,
                              cudaStream_t stream) {
    if (!q_t) {
        launch_pdl(quantize_row_kernel<FMT>, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0, stream, xs, cols, pow2, q, scale_inv);
        return cudaGetLastError();
    }
    // with the transposed copy: two tiled reads of x; the scale arrays hold the
    // row / column maxima until the last step turns them into 1/scale
    const cudaError_t e = launch_zero(scale_inv, rows, scale_inv_t, cols, stream);
    if (e != cudaSuccess) return e;
    const int64_t tiles_c = (cols + 127) / 128, tiles = ((rows + 127) / 128) * tiles_c;
    auto* rmax = reinterpret_cast<unsigned*>(scale_inv);
    auto* cmax = reinterpret_cast<unsigned*>(scale_inv_t);
    const int group = tiles >= 8 * static_cast<int64_t>(num_sms()) ? 4 : 1;
    const int64_t groups_r = ((rows + 127) / 128 + group - 1) / group;
    launch_pdl(row_col_amax_kernel, dim3(static_cast<unsigned>(groups_r * tiles_c)), dim3(kThreads),
               0, stream, xs, rows, cols, tiles_c, group, rmax, cmax);
    launch_pdl(quantize_row_col_kernel<FMT>, dim3(static_cast<unsigned>(tiles)), dim3(kThreads), 0, stream, 
        xs, rows, cols, tiles_c, pow2, rmax, cmax, q, q_t);
    launch_pdl(row_col_scale_finalize_kernel<FMT>, dim3(static_cast<unsigned>((rows + cols + 255) / 256)),
               dim3(256), 0, stream, scale_inv, rows, scale_inv_t, cols, pow2);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* x, int64_t rows, int64_t cols, int fmt, int pow2,
                                 uint8_t* q, float* scale_inv, uint8_t* q_t, float* scale_inv_t,
                                 cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const uint16_t* xs = static_cast<const uint16_t*>(x);
    return fmt == 0 ? launch_row<0>(xs, rows, cols, pow2, q, scale_inv, q_t, scale_inv_t, stream)
                    : launch_row<1>(xs, rows, cols, pow2, q, scale_inv, q_t, scale_inv_t, stream);
}

// The dual cast's dynamic shared-memory limit, set once per device and format.
template <typename Kernel>
cudaError_t dual_smem_attr(Kernel k, int fmt) {
    static std::mutex mu;
    static bool done[64][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    const bool cached = dev >= 0 && dev < 64;
    std::lock_guard<std::mutex> lock(mu);
    if (cached && done[dev][fmt]) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kDualSmem);
    if (e == cudaSuccess && cached) done[dev][fmt] = true;
    return e;
}

cudaError_t launch_quantize_block(const void* x, int64_t rows, int64_t cols, int fmt, int gran,
                                  int pow2, uint8_t* q, float* scale_inv, uint8_t* q_t,
                                  float* scale_inv_t, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const uint16_t* xs = static_cast<const uint16_t*>(x);
    if (gran == 1 && q_t) {
        const int64_t tiles_c = cols / 128;
        const unsigned tiles = static_cast<unsigned>((rows / 128) * tiles_c);
        CUtensorMap tmX;
        if (make_bf16_box_map(&tmX, x, rows, cols, 128, 128) != FP8_OK) return cudaErrorInvalidValue;
        auto k = fmt == 0 ? quantize_1x128_dual_kernel<0> : quantize_1x128_dual_kernel<1>;
        const cudaError_t e = dual_smem_attr(k, fmt);
        if (e != cudaSuccess) return e;
        const int64_t ctas = 2 * static_cast<int64_t>(num_sms());
        const unsigned grid = static_cast<unsigned>(tiles < ctas ? tiles : ctas);
        launch_pdl(k, dim3(grid), dim3(kThreads), kDualSmem, stream, tmX, rows, cols, tiles_c,
                   static_cast<int64_t>(tiles), pow2, q, scale_inv, q_t, scale_inv_t,
                   device_status_word());
    } else if (gran == 1) {
        const int64_t pairs = (rows * (cols / 128) + 1) / 2;
        const int grid = grid_for(pairs, kThreads / 32);
        if (fmt == 0) launch_pdl(quantize_1x128_kernel<0>, dim3(grid), dim3(kThreads), 0, stream, xs, rows, cols, pow2, q, scale_inv);
        else launch_pdl(quantize_1x128_kernel<1>, dim3(grid), dim3(kThreads), 0, stream, xs, rows, cols, pow2, q, scale_inv);
    } else {
        const unsigned tiles = static_cast<unsigned>((rows / 128) * (cols / 128));
        if (fmt == 0) launch_pdl(quantize_128x128_kernel<0>, dim3(tiles), dim3(kThreads), 0, stream, xs, rows, cols, pow2, q, scale_inv, q_t, scale_inv_t);
        else launch_pdl(quantize_128x128_kernel<1>, dim3(tiles), dim3(kThreads), 0, stream, xs, rows, cols, pow2, q, scale_inv, q_t, scale_inv_t);
    }
    return cudaGetLastError();
}

}  // namespace fp8
