/*
 * fp8_oracle.c -- plain CPU oracle for the scaled FP8 linear layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the package
 * smoke check and the benchmark's CPU-baseline leg may load this library.
 * It shares no code, header, table or constant generator with the CUDA path
 * in scaled_fp8_linear_gb300/csrc; each side is written from the format and
 * scaling definitions on its own.
 *
 * Everything here is the slow, obvious definition:
 *   - FP8 codes are decoded from their bit fields and encoded by exact integer
 *     arithmetic on the fp32 bit pattern (no floating rounding tricks);
 *   - amax is an integer max over |bf16| bit patterns (exact, order-free);
 *   - the scale update follows the delayed/history recipe step by step;
 *   - GEMMs sum exact fp64 products of decoded codes in fp64.
 *
 * Sources (page titles; sections):
 *   [MP]  "Mixed Precision LLM Training: The Complete Guide"
 *         - "The precision formats" table and "FP8 E4M3" / "FP8 E5M2"
 *           (bit layouts, ranges ~2^-9..448 and ~2^-16..57344);
 *         - "Transformer Engine internals" > "Per-tensor scaling",
 *           "Delayed scaling", "History-based scaling", "The HYBRID recipe",
 *           "Skipping the BAcc accumulator promotion";
 *         - "DeepSeek FP8 training recipe" > "Block-wise scaling at 128
 *           granularity", "Mixed-precision accumulation";
 *         - "torch.compile and FP8" (skip the scale update for an all-zero
 *           tensor);
 *         - "Calibration deep dive" > "Dynamic calibration" (margin,
 *           amax_history_len, amax_compute_algo "max" / "most_recent").
 *   [TI]  "Training and inference of large language models using 8-bit
 *         floating point" (abstract: per-tensor scales updated dynamically;
 *         reviews: per-tensor "scaling bias", i.e. power-of-two scales).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (see build.py).
 * -ffp-contract=off keeps every float multiply a single IEEE rounding.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

#define ORC_ALGO_MAX 0
#define ORC_ALGO_MOST_RECENT 1

#define ORC_GRAN_TENSOR 0
#define ORC_GRAN_1x128 1
#define ORC_GRAN_128x128 2
#define ORC_GRAN_ROW 3

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 is the top half of an fp32 bit pattern: widening is exact. */
float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------------ codec */

/* [MP] "FP8 E4M3" / "FP8 E5M2": 1 sign bit, E exponent bits, M mantissa bits.
 * Normal:    (-1)^S * 2^(e - bias) * (1 + m / 2^M),   e > 0
 * Subnormal: (-1)^S * 2^(1 - bias) * (m / 2^M),       e = 0
 * E4M3 (bias 7): the all-ones code S.1111.111 is NaN and there is no Inf
 * (the "fn" variant, torch.float8_e4m3fn); largest finite 1.75*2^8 = 448,
 * smallest subnormal 2^-9.
 * E5M2 (bias 15): exponent 31 with m = 0 is Inf, m != 0 is NaN; largest
 * finite 1.75*2^15 = 57344, smallest subnormal 2^-16. */
double orc_decode(uint8_t c, int fmt)
{
    const double sign = (c & 0x80) ? -1.0 : 1.0;
    if (fmt == ORC_E4M3) {
        int e = (c >> 3) & 0xF, m = c & 0x7;
        if (e == 15 && m == 7) return NAN;
        if (e == 0) return sign * ldexp((double)m / 8.0, 1 - 7);
        return sign * ldexp(1.0 + (double)m / 8.0, e - 7);
    } else {
        int e = (c >> 2) & 0x1F, m = c & 0x3;
        if (e == 31) return m == 0 ? sign * INFINITY : NAN;
        if (e == 0) return sign * ldexp((double)m / 4.0, 1 - 15);
        return sign * ldexp(1.0 + (double)m / 4.0, e - 15);
    }
}

/* Largest finite code (positive): E4M3 0.1111.110 = 448, E5M2 0.11110.11 = 57344. */
static uint8_t max_code(int fmt) { return fmt == ORC_E4M3 ? 0x7E : 0x7B; }

double orc_fp8_max(int fmt) { return orc_decode(max_code(fmt), fmt); }

/* Encode one fp32 value, round-to-nearest-even, saturating to the largest
 * finite value ("satfinite"): NaN -> canonical NaN 0x7F; +-Inf and every
 * |v| above the largest finite value -> +-max; underflow keeps the sign.
 * The rounding is done on integers: |v| = sig * 2^e2 exactly, the target
 * grid spacing in the binade of |v| is 2^qe, and sig is divided by
 * 2^(qe - e2) with an explicit round-half-to-even on the remainder. */
uint8_t orc_encode(float v, int fmt)
{
    const int mb = (fmt == ORC_E4M3) ? 3 : 2;      /* mantissa bits        */
    const int bias = (fmt == ORC_E4M3) ? 7 : 15;   /* exponent bias        */
    const int emin = 1 - bias;                     /* min normal exponent  */
    const uint32_t u = f32_bits(v);
    const uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    const uint32_t ex = (u >> 23) & 0xFF, fr = u & 0x7FFFFF;

    if (ex == 0xFF) return fr ? 0x7F : (uint8_t)(sign | max_code(fmt));
    if (ex == 0 && fr == 0) return sign;

    uint64_t sig;
    int e2;
    if (ex == 0) { sig = fr; e2 = -149; }           /* fp32 subnormal */
    else { sig = fr | 0x800000u; e2 = (int)ex - 150; }
    int top = 63;
    while (!((sig >> top) & 1u)) --top;
    const int E = e2 + top;                          /* |v| in [2^E, 2^(E+1)) */

    int qe = (E > emin ? E : emin) - mb;             /* grid spacing 2^qe */
    const int shift = qe - e2;                       /* >= 1 for fp32 input */
    uint64_t n;
    if (shift <= 0) {
        n = sig << (-shift);
    } else if (shift > 40) {
        n = 0;                                       /* far below half a step */
    } else {
        n = sig >> shift;
        const uint64_t rem = sig & ((1ull << shift) - 1);
        const uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;
    }
    if (n == 0) return sign;
    if (n == (1ull << (mb + 1))) { n >>= 1; qe += 1; } /* carried into next binade */

    if (n < (1ull << mb)) return (uint8_t)(sign | n);  /* subnormal */
    const int field = qe + mb + bias;
    const uint64_t man = n - (1ull << mb);
    if (fmt == ORC_E4M3) {
        if (field > 15 || (field == 15 && man == 7)) return (uint8_t)(sign | max_code(fmt));
        return (uint8_t)(sign | (field << 3) | man);
    } else {
        if (field > 30) return (uint8_t)(sign | max_code(fmt));
        return (uint8_t)(sign | (field << 2) | man);
    }
}

void orc_decode_array(const uint8_t* c, int64_t n, int fmt, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode(c[i], fmt);
}

void orc_encode_array(const float* v, int64_t n, int fmt, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode(v[i], fmt);
}

/* ------------------------------------------------------------------- amax */

/* max |x| over a bf16 tensor.  |x| of a bf16 is its bit pattern with the
 * sign cleared, and for non-negative floats the bit patterns order like the
 * values, so the max is an integer max: exact and independent of order.
 * Any NaN gives a NaN (its |bits| exceed those of +Inf). */
float orc_amax_bf16(const uint16_t* x, int64_t n)
{
    uint16_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint16_t a = x[i] & 0x7FFF;
        if (a > m) m = a;
    }
    return orc_bf16_to_f32(m);
}

/* ------------------------------------------------------------ scale update */

/* One scale from one effective amax, the rule shared by the per-tensor and
 * the block recipes ([MP] "Per-tensor scaling": the scale puts the tensor's
 * max |x| at the top of the FP8 range):
 *   s = fp8_max / amax              (one fp32 IEEE division)
 *   s = s * 2^-margin               (one fp32 multiply by an exact power of 2)
 *   s clamped to [FLT_MIN, FLT_MAX] (the scale "floor" and ceiling; keeps
 *                                    1/s finite)
 *   pow2: s = 2^floor(log2 s)       ([TI] exponent-bias scaling), done by
 *                                    clearing the fp32 mantissa bits. */
static float scale_from_amax(float amax, int fmt, int margin, int pow2)
{
    float s = (float)orc_fp8_max(fmt) / amax;
    s = s * ldexpf(1.0f, -margin);
    if (!(s <= FLT_MAX)) s = FLT_MAX;
    if (s < FLT_MIN) s = FLT_MIN;
    if (pow2) s = bits_f32(f32_bits(s) & 0xFF800000u);
    return s;
}

/* Delayed / history scaling ([MP] "Delayed scaling", "History-based
 * scaling", "Dynamic calibration"):
 *   1. history[pos] = amax;  pos = (pos + 1) mod H
 *   2. amax_eff = max(history)   for algo "max"
 *                 amax           for algo "most_recent"
 *   3. if amax_eff is zero or not finite, scale and scale_inv stay as they
 *      are ([MP] "torch.compile and FP8": the update is skipped for an
 *      all-zero tensor);
 *      else scale = scale_from_amax(amax_eff), scale_inv = 1 / scale.
 * Dynamic (current) scaling is the same rule with H = 1.  The scale that
 * this produces is used for the NEXT quantization (one-step lag). */
void orc_update_scale(float amax, float* history, int32_t* pos, int H, int algo,
                      int fmt, int margin, int pow2, float* scale, float* scale_inv)
{
    history[*pos] = amax;
    *pos = (*pos + 1) % H;
    float eff;
    if (algo == ORC_ALGO_MOST_RECENT) {
        eff = amax;
    } else {
        eff = history[0];
        for (int i = 1; i < H; ++i)
            if (isnan(history[i]) || history[i] > eff) eff = history[i];
    }
    if (!(eff > 0.0f) || !isfinite(eff)) return;
    const float s = scale_from_amax(eff, fmt, margin, pow2);
    *scale = s;
    *scale_inv = 1.0f / s;
}

/* ------------------------------------------------------ stochastic rounding */

/* Philox-4x32-10, the counter-based generator of Salmon, Moraes, Dror and
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of
 *   (c0,c1,c2,c3) -> (hi(B*c2)^c1^k0, lo(B*c2), hi(A*c0)^c3^k1, lo(A*c0))
 * with A = 0xD2511F53, B = 0xCD9E8D57, the key bumped by the Weyl constants
 * (0x9E3779B9, 0xBB67AE85) between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Stochastic rounding of one fp32 value onto the FP8 grid ([MP] "Stochastic
 * rounding": round up or down at random, in proportion to the remainder):
 * |v| = sig * 2^e2 lies between the grid points n*2^qe and (n+1)*2^qe with
 * remainder rem = sig mod 2^shift (shift = qe - e2); the magnitude is rounded
 * up iff r32 < floor(rem * 2^32 / 2^shift), r32 a uniform 32-bit draw, so a
 * value rounds up with probability rem/2^shift (exactly, for shift <= 32).
 * NaN, infinities, saturation and signed zeros as in orc_encode. */
uint8_t orc_encode_sr(float v, int fmt, uint32_t r32)
{
    const int mb = (fmt == ORC_E4M3) ? 3 : 2;
    const int bias = (fmt == ORC_E4M3) ? 7 : 15;
    const int emin = 1 - bias;
    const uint32_t u = f32_bits(v);
    const uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    const uint32_t ex = (u >> 23) & 0xFF, fr = u & 0x7FFFFF;
    if (ex == 0xFF) return fr ? 0x7F : (uint8_t)(sign | max_code(fmt));
    if (ex == 0 && fr == 0) return sign;
    uint64_t sig;
    int e2;
    if (ex == 0) { sig = fr; e2 = -149; }
    else { sig = fr | 0x800000u; e2 = (int)ex - 150; }
    int top = 63;
    while (!((sig >> top) & 1u)) --top;
    const int E = e2 + top;
    int qe = (E > emin ? E : emin) - mb;
    const int shift = qe - e2;                     /* >= 1 */
    uint64_t n, threshold;
    if (shift >= 56) {
        n = 0;                                     /* sig < 2^24: rem * 2^32 / 2^shift < 1 */
        threshold = 0;
    } else {
        n = sig >> shift;
        const uint64_t rem = sig & ((1ull << shift) - 1);
        threshold = shift <= 32 ? rem << (32 - shift) : rem >> (shift - 32);
    }
    if ((uint64_t)r32 < threshold) n += 1;
    if (n == 0) return sign;
    if (n == (1ull << (mb + 1))) { n >>= 1; qe += 1; }
    if (n < (1ull << mb)) return (uint8_t)(sign | n);
    const int field = qe + mb + bias;
    const uint64_t man = n - (1ull << mb);
    if (fmt == ORC_E4M3) {
        if (field > 15 || (field == 15 && man == 7)) return (uint8_t)(sign | max_code(fmt));
        return (uint8_t)(sign | (field << 3) | man);
    } else {
        if (field > 30) return (uint8_t)(sign | max_code(fmt));
        return (uint8_t)(sign | (field << 2) | man);
    }
}

/* Per-tensor cast with stochastic rounding: element i (row-major index) uses
 * word (i mod 4) of Philox(counter = (lo(i/4), hi(i/4), lo(offset),
 * hi(offset)), key = (lo(seed), hi(seed))).  q_t (nullable) = transpose. */
void orc_quantize_sr(const uint16_t* x, int64_t rows, int64_t cols, int fmt, float scale,
                     uint64_t seed, uint64_t offset, uint8_t* q, uint8_t* qt)
{
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            const uint64_t idx = (uint64_t)(i * cols + j);
            const uint64_t g = idx >> 2;
            const uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset,
                                     (uint32_t)(offset >> 32)};
            uint32_t r[4];
            orc_philox4x32_10(ctr, key, r);
            const float v = orc_bf16_to_f32(x[idx]) * scale;
            const uint8_t c = orc_encode_sr(v, fmt, r[idx & 3]);
            if (q) q[idx] = c;
            if (qt) qt[j * rows + i] = c;
        }
    }
}

/* --------------------------------------------------------------- quantize */

/* [MP] "Per-tensor scaling": multiply by the scale, then cast to FP8.
 *   q[i][j]  = encode(fp32(x[i][j]) * s)   (one fp32 multiply, RNE, satfinite)
 *   qt[j][i] = q[i][j]                     (optional transposed copy) */
void orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int fmt, float scale,
                  uint8_t* q, uint8_t* qt)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            const float v = orc_bf16_to_f32(x[i * cols + j]) * scale;
            const uint8_t c = orc_encode(v, fmt);
            if (q) q[i * cols + j] = c;
            if (qt) qt[j * rows + i] = c;
        }
    }
}

/* Dashboard counters of a per-tensor cast ([MP] "Numerical-failure taxonomy"
 * > "A diagnostic dashboard": underflow ratio, saturation), over the cast of
 * orc_quantize with the same scale:
 *   counts[0] = inputs x != +-0 whose FP8 code is +-0     (flushed to zero)
 *   counts[1] = inputs whose scaled value |fp32(x) * s| is above the largest
 *               finite FP8 value (so the cast saturates; +-Inf included,
 *               NaN not) */
void orc_cast_counts(const uint16_t* x, int64_t n, int fmt, float scale, uint64_t* counts)
{
    const float fmax = (float)orc_fp8_max(fmt);
    uint64_t under = 0, sat = 0;
    for (int64_t i = 0; i < n; ++i) {
        const float v = orc_bf16_to_f32(x[i]) * scale;
        const uint8_t c = orc_encode(v, fmt);
        if ((x[i] & 0x7FFF) != 0 && (c & 0x7F) == 0) ++under;
        if (fabsf(v) > fmax) ++sat;
    }
    counts[0] = under;
    counts[1] = sat;
}

/* [MP] "Block-wise scaling at 128 granularity": one scale per 1x128 segment
 * of a row (activations, gradients) or per 128x128 tile (weights).  Each
 * block's scale comes from its own amax with margin 0 and no history; an
 * all-zero (or non-finite) block gets scale 1.  scale_inv[bi][bj] = 1/s for
 * block row bi (= row for 1x128, row/128 for 128x128) and block column bj =
 * col/128, row-major [rows/block_rows][cols/128]. */
void orc_block_quantize(const uint16_t* x, int64_t rows, int64_t cols, int fmt,
                        int block_rows, int pow2, uint8_t* q, float* scale_inv)
{
    const int64_t nbr = rows / block_rows, nbc = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t bi = 0; bi < nbr; ++bi) {
        for (int64_t bj = 0; bj < nbc; ++bj) {
            uint16_t m = 0;
            for (int64_t i = bi * block_rows; i < (bi + 1) * block_rows; ++i)
                for (int64_t j = bj * 128; j < (bj + 1) * 128; ++j) {
                    uint16_t a = x[i * cols + j] & 0x7FFF;
                    if (a > m) m = a;
                }
            const float amax = orc_bf16_to_f32(m);
            float s = 1.0f;
            if (amax > 0.0f && isfinite(amax)) s = scale_from_amax(amax, fmt, 0, pow2);
            scale_inv[bi * nbc + bj] = 1.0f / s;
            for (int64_t i = bi * block_rows; i < (bi + 1) * block_rows; ++i)
                for (int64_t j = bj * 128; j < (bj + 1) * 128; ++j)
                    q[i * cols + j] = orc_encode(orc_bf16_to_f32(x[i * cols + j]) * s, fmt);
        }
    }
}

/* Per-row (per-channel) scaling ([MP] "Transformer Engine internals" >
 * "Per-row vs per-tensor scaling"; "Calibration deep dive" > "Per-channel vs
 * per-tensor"): every row of x gets its own scale from its own amax, by the
 * block rule with the whole row as the block (margin 0; 1 for an all-zero or
 * non-finite row; optional power of two).  scale_inv [rows]. */
void orc_row_quantize(const uint16_t* x, int64_t rows, int64_t cols, int fmt, int pow2,
                      uint8_t* q, float* scale_inv)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        uint16_t m = 0;
        for (int64_t j = 0; j < cols; ++j) {
            uint16_t a = x[i * cols + j] & 0x7FFF;
            if (a > m) m = a;
        }
        const float amax = orc_bf16_to_f32(m);
        float s = 1.0f;
        if (amax > 0.0f && isfinite(amax)) s = scale_from_amax(amax, fmt, 0, pow2);
        scale_inv[i] = 1.0f / s;
        for (int64_t j = 0; j < cols; ++j)
            q[i * cols + j] = orc_encode(orc_bf16_to_f32(x[i * cols + j]) * s, fmt);
    }
}

/* ------------------------------------------------------------------- GEMM */

/* Dequantisation factor of operand row r for K-block kb under a granularity:
 * per-tensor: s[0]; 1x128: s[r*KB + kb]; 128x128: s[(r/128)*KB + kb]. */
static double factor(const float* s, int gran, int64_t r, int64_t kb, int64_t KB)
{
    if (gran == ORC_GRAN_TENSOR) return (double)s[0];
    if (gran == ORC_GRAN_ROW) return (double)s[r];
    if (gran == ORC_GRAN_1x128) return (double)s[r * KB + kb];
    return (double)s[(r / 128) * KB + kb];
}

/* One output entry of the scaled FP8 GEMM ("TN": A [M x K] and B [N x K],
 * both row-major with K contiguous):
 *   per-tensor: D[i][j] = (sa * sb) * sum_k dec(A[i][k]) * dec(B[j][k])
 *   block:      D[i][j] = sum_kb sa(i,kb) * sb(j,kb) * sum_{k in kb} dec(A)dec(B)
 * where sa, sb are the dequantisation factors (1 / quantisation scale); a
 * per-row factor (sa[i] or sb[j]) is used like a per-tensor one.  The
 * products of two FP8 values are exact in fp64 and are summed in fp64
 * ([MP] "Skipping the BAcc accumulator promotion": FP8 is the multiplicand
 * precision, the accumulator is wider).  Dabs is the same sum over |terms|,
 * the denominator of the error bound. */
static void gemm_entry(const double* ta, const double* tb, const uint8_t* A, const uint8_t* B,
                       int64_t K, int64_t i, int64_t j, int ga, const float* sa, int gb,
                       const float* sb, double* d, double* dabs)
{
    const uint8_t* a = A + i * K;
    const uint8_t* b = B + j * K;
    if ((ga == ORC_GRAN_TENSOR || ga == ORC_GRAN_ROW) && (gb == ORC_GRAN_TENSOR || gb == ORC_GRAN_ROW)) {
        /* per-tensor or per-row factors do not vary along k: outside the sum */
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p = ta[a[k]] * tb[b[k]];
            acc += p;
            aacc += fabs(p);
        }
        const double f = factor(sa, ga, i, 0, 1) * factor(sb, gb, j, 0, 1);
        *d = f * acc;
        *dabs = fabs(f) * aacc;
        return;
    }
    const int64_t KB = K / 128;
    double acc = 0.0, aacc = 0.0;
    for (int64_t kb = 0; kb < KB; ++kb) {
        double part = 0.0, apart = 0.0;
        for (int64_t k = kb * 128; k < (kb + 1) * 128; ++k) {
            const double p = ta[a[k]] * tb[b[k]];
            part += p;
            apart += fabs(p);
        }
        const double f = factor(sa, ga, i, kb, KB) * factor(sb, gb, j, kb, KB);
        acc += f * part;
        aacc += fabs(f) * apart;
    }
    *d = acc;
    *dabs = aacc;
}

static void decode_table(int fmt, double* t)
{
    for (int c = 0; c < 256; ++c) t[c] = orc_decode((uint8_t)c, fmt);
}

/* Full output D [M x N] (row-major). */
void orc_gemm(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t M, int64_t N,
              int64_t K, int ga, const float* sa, int gb, const float* sb, double* D,
              double* Dabs)
{
    double ta[256], tb[256];
    decode_table(fa, ta);
    decode_table(fb, tb);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            gemm_entry(ta, tb, A, B, K, i, j, ga, sa, gb, sb, &D[i * N + j], &Dabs[i * N + j]);
}

/* Selected entries (ii[t], jj[t]) of D, for outputs too large to compute whole. */
void orc_gemm_entries(const uint8_t* A, int fa, const uint8_t* B, int fb, int64_t K, int ga,
                      const float* sa, int gb, const float* sb, const int64_t* ii,
                      const int64_t* jj, int64_t count, double* D, double* Dabs)
{
    double ta[256], tb[256];
    decode_table(fa, ta);
    decode_table(fb, tb);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t t = 0; t < count; ++t)
        gemm_entry(ta, tb, A, B, K, ii[t], jj[t], ga, sa, gb, sb, &D[t], &Dabs[t]);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
