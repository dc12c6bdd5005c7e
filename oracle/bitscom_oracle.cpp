/*
 * bitscom_oracle.cpp -- plain, slow, single-threaded CPU oracle of the
 * low-bit gradient codec.  TEST INFRASTRUCTURE ONLY (see the header): only
 * the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * Written for obviousness, not speed: one element at a time, one bit at a
 * time when packing, recursion for the tree sum.  Build flags must keep IEEE
 * single precision exact:  -O2 -ffp-contract=off -fno-fast-math
 * (no fused multiply-add contraction, no reassociation, no flush to zero).
 *
 * Sources of each rule:
 *  - bitwidths {1,2,4,8,12,16}, quantize / dequantize, bit-packing,
 *    stochastic rounding, per-block FP16 scales, first-stage error feedback,
 *    stage2_error_feedback: bitscom README, "Implemented Features" and
 *    "Backend Registration Options".
 *  - the reduce sits between an all-to-all and an all-gather: bitscom README,
 *    "Implemented Features" (low-bit all-reduce pipeline); the decoupled
 *    reduce-scatter + all-gather structure: DeAR README, opening paragraph.
 *  - exact arithmetic (the pages state none): symmetric absmax scaling with
 *    Qmax = 2^(b-1)-1, fp32 correctly rounded division, round half to even,
 *    1-bit sign with a mean-magnitude scale, Philox4x32-10 keyed by (seed,
 *    element index), offset-binary codes packed LSB-first, e' = (g+e) - s*q.
 *    The readings of every step the pages leave open are listed beside the
 *    function that takes them.
 */
#include "bitscom_oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 / bfloat16 conversions from the format definitions */
/* ------------------------------------------------------------------ */

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float float_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary32 -> binary16, round to nearest, ties to even, with gradual
 * underflow (fp16 subnormals kept) and overflow to infinity.
 * A finite binary32 value is m * 2^E with m < 2^24.  The binary16 result is
 * M * 2^F with F = e16 - 25 for a normal (M in [2^10, 2^11)) or F = -24 for a
 * subnormal (M < 2^10).  Pick F from the magnitude, shift m right by F - E
 * with round-half-even, and re-normalise if the rounding carried. */
uint16_t orc_f32_to_f16(float x)
{
    uint32_t u = bits_of(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t e = (u >> 23) & 0xFFu;
    uint32_t frac = u & 0x7FFFFFu;
    if (e == 0xFFu) {                     /* inf or NaN */
        if (frac == 0) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u); /* NaN: outside the codec's domain */
    }
    uint64_t m = (e == 0) ? frac : (frac | 0x800000u);
    if (m == 0) return sign;
    int E = (e == 0 ? 1 : (int)e) - 127 - 23;
    int top = 63 - __builtin_clzll(m);    /* floor(log2(m)) */
    int F = E + top - 10;                 /* keep 11 significant bits */
    if (F < -24) F = -24;                 /* binary16 subnormal spacing */
    int sh = F - E;
    uint64_t M;
    if (sh <= 0) {
        M = m << (-sh);
    } else if (sh > 40) {
        M = 0;                            /* far below half of 2^-24 */
    } else {
        M = m >> sh;
        uint64_t rem = m - (M << sh);
        uint64_t half = (uint64_t)1 << (sh - 1);
        if (rem > half || (rem == half && (M & 1u))) M += 1;
    }
    if (M == 2048) { M = 1024; F += 1; }  /* rounding carried into a new binade */
    if (M < 1024) return (uint16_t)(sign | (uint16_t)M);   /* subnormal (F == -24) */
    int e16 = F + 25;
    if (e16 >= 31) return (uint16_t)(sign | 0x7C00u);      /* overflow */
    return (uint16_t)(sign | (uint16_t)(e16 << 10) | (uint16_t)(M - 1024));
}

float orc_f16_to_f32(uint16_t h)
{
    int sign = (h & 0x8000u) ? -1 : 1;
    int e16 = (h >> 10) & 31;
    int frac = h & 1023;
    if (e16 == 31) return frac ? NAN : sign * INFINITY;
    if (e16 == 0) return sign * ldexpf((float)frac, -24);
    return sign * ldexpf((float)(1024 + frac), e16 - 25);
}

float orc_bf16_to_f32(uint16_t b) { return float_of((uint32_t)b << 16); }

/* binary32 -> bfloat16, round to nearest even: keep the top 16 bits and
 * round on the 16 dropped ones (ties to an even kept part); a carry out of the
 * mantissa moves into the exponent, so the largest finite values overflow to
 * infinity exactly as IEEE rounding does.  NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = bits_of(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t kept = u >> 16, dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1;
    return (uint16_t)kept;
}

void orc_f32_to_f16_many(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as  */
/* 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies; the key    */
/* is bumped by the Weyl constants between rounds.                      */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Reading of "keyed by (seed, element index)": key = the two 32-bit halves of
 * the seed; counter = (low, high halves of i/4, stream, 0); element i takes
 * output word i mod 4, so one Philox call serves four consecutive elements. */
uint32_t orc_random_word(uint64_t seed, uint32_t stream, uint64_t i)
{
    uint64_t g = i >> 2;
    uint32_t ctr[4] = { (uint32_t)g, (uint32_t)(g >> 32), stream, 0u };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[i & 3];
}

void orc_random_words(uint64_t seed, uint32_t stream, uint64_t i0, int64_t n, uint32_t* out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = orc_random_word(seed, stream, i0 + (uint64_t)k);
}

/* ------------------------------------------------------------------ */
/* Scalar rules                                                         */
/* ------------------------------------------------------------------ */

static int valid_bits(int b) { return b == 1 || b == 2 || b == 4 || b == 8 || b == 12 || b == 16; }
static int valid_block(int B) { return B >= 8 && (B & (B - 1)) == 0; }
/* Reading of the SDP4Bit README's "--hadamard-transform" (TLq-HS): a
 * Walsh-Hadamard rotation of every H-element block before quantisation and
 * its inverse after dequantisation; H is a power of two in [8, 256] dividing
 * the quantisation block, and every stage of one all-reduce uses the same H. */
static int valid_hadamard(int H, int B)
{
    return H == 0 || (H >= 8 && H <= 256 && (H & (H - 1)) == 0 && B % H == 0);
}

static int valid_params(const orc_params* p)
{
    return p && valid_bits(p->bits) && valid_block(p->block) &&
           (p->rounding == 0 || p->rounding == 1) && valid_hadamard(p->hadamard, p->block);
}

/* Sylvester-ordered unnormalised Walsh-Hadamard transform of one block: stage
 * h = 1, 2, 4, ... replaces (x[j], x[j+h]) by (x[j] + x[j+h], x[j] - x[j+h])
 * for every j whose bit h is clear; each output is one fp32 operation, so the
 * result does not depend on the order within a stage.  Applying it twice
 * gives H times the input (up to rounding). */
static void fwht_block(float* x, int H)
{
    for (int h = 1; h < H; h *= 2)
        for (int i = 0; i < H; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
}

int orc_fwht(float* x, int64_t n, int32_t H)
{
    if (!x || H < 1 || (H & (H - 1)) != 0 || n < 0 || n % H != 0) return 1;
    for (int64_t k = 0; k < n; k += H) fwht_block(x + k, H);
    return 0;
}

int64_t orc_num_blocks(int64_t n, int32_t block) { return (n + block - 1) / block; }
int64_t orc_packed_bytes(int64_t n, int32_t bits, int32_t block)
{
    return orc_num_blocks(n, block) * block * bits / 8;
}

/* Round half to even, written from its definition. */
static float round_half_even(float t)
{
    float f = floorf(t);
    /* t - f is exact except for -1 < t < 0, where it rounds 1 + t; that
     * rounding is monotone and 0.5 is representable, so the comparisons
     * below still pick the right neighbour. */
    float frac = t - f;
    if (frac > 0.5f) return f + 1.0f;
    if (frac < 0.5f) return f;
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Balanced binary tree over contiguous halves: sum(a[0:n]) =
 * sum(a[0:n/2]) + sum(a[n/2:n]), n a power of two.  This fixes the fp32
 * summation order of the 1-bit mean so that any implementation can match it. */
static float tree_sum(const float* a, int64_t n)
{
    if (n == 1) return a[0];
    return tree_sum(a, n / 2) + tree_sum(a + n / 2, n / 2);
}

/* Scale of one block of magnitudes |v| (already zero-padded to B).
 * b >= 2 : s = fp16(min(absmax / Qmax, 65504)), fp32 division correctly
 *          rounded (the per-block FP16 scale of "Implemented Features").
 * b == 1 : s = fp16(min(mean |v|, 65504)), mean = tree_sum / n_valid.
 * The clamp to the largest finite fp16 is a reading: the pages do not say
 * what happens on overflow. */
static uint16_t block_scale(const float* absv, int B, int n_valid, int bits)
{
    float x;
    if (bits == 1) {
        float sum = tree_sum(absv, B);
        x = sum / (float)n_valid;
    } else {
        float amax = 0.0f;
        for (int j = 0; j < B; ++j) if (absv[j] > amax) amax = absv[j];
        float qmax = (float)((1 << (bits - 1)) - 1);
        x = amax / qmax;
    }
    if (x > 65504.0f) x = 65504.0f;
    return orc_f32_to_f16(x);
}

/* Integer code q of one value v under scale s (fp32 value of the fp16 scale).
 * b >= 2, round half to even : q = clamp(rint(v/s), -Qmax, Qmax)
 * b >= 2, stochastic         : t = v/s, f = floor(t), p = t - f (exact,
 *                              not rounded to fp32), u = (r mod 2^23) * 2^-23
 *                              with r the element's Philox word,
 *                              q = clamp(f + [u < p], +-Qmax)
 * s == 0 gives q = 0 (reading: an all-zero or underflowed block).
 * b == 1 : q = +1 if v >= 0 else -1 (reading: +0 and -0 both map to +1; the
 *          rounding mode is ignored, the 1-bit code is a deterministic sign). */
static int32_t quantize_value(float v, float s, const orc_params* p, uint64_t gindex)
{
    int b = p->bits;
    if (b == 1) return (v >= 0.0f) ? 1 : -1;
    float qmax = (float)((1 << (b - 1)) - 1);
    if (s == 0.0f) return 0;
    float t = v / s;
    float q;
    if (p->rounding == 0) {
        q = round_half_even(t);
    } else {
        uint32_t r = orc_random_word(p->seed, p->philox_stream, gindex);
        float u = (float)(r & 0x7FFFFFu) * (1.0f / 8388608.0f);
        float f = floorf(t);
        /* Round up iff u < t - f, the fraction taken exactly: u < t - f is
         * f + u < t, and f + u is exact in fp64 while |t| < 2^23 (an integer
         * of at most 24 bits plus a multiple of 2^-23).  Larger t are
         * integers (t = f), and the rounded f + u is never below f. */
        q = f + (((double)f + (double)u < (double)t) ? 1.0f : 0.0f);
    }
    q = clampf(q, -qmax, qmax);
    return (int32_t)q;
}

/* Offset-binary code: u = q + 2^(b-1) for b >= 2; u = (q + 1) / 2 for b = 1. */
static uint32_t offset_code(int32_t q, int bits)
{
    if (bits == 1) return (uint32_t)((q + 1) / 2);
    return (uint32_t)(q + (1 << (bits - 1)));
}

static int32_t code_to_q(uint32_t u, int bits)
{
    if (bits == 1) return (int32_t)(2 * u) - 1;
    return (int32_t)u - (1 << (bits - 1));
}

/* LSB-first bit stream: bit k of the stream is bit (k mod 8) of byte k/8;
 * element e's code occupies stream bits [e*b, e*b + b), least significant
 * bit first.  Little-endian 32-bit words of this stream are the same bytes. */
static void put_code(uint8_t* stream, int64_t e, int bits, uint32_t u)
{
    for (int k = 0; k < bits; ++k) {
        int64_t pos = e * bits + k;
        uint8_t bit = (uint8_t)((u >> k) & 1u);
        stream[pos / 8] = (uint8_t)((stream[pos / 8] & ~(1u << (pos % 8))) | (bit << (pos % 8)));
    }
}

static uint32_t get_code(const uint8_t* stream, int64_t e, int bits)
{
    uint32_t u = 0;
    for (int k = 0; k < bits; ++k) {
        int64_t pos = e * bits + k;
        u |= (uint32_t)((stream[pos / 8] >> (pos % 8)) & 1u) << k;
    }
    return u;
}

/* ------------------------------------------------------------------ */
/* One quantisation stage over an fp32 vector v (shared by the encoder   */
/* and the decoder's requantisation).                                   */
/* ------------------------------------------------------------------ */

/* Quantise v[0:n) block by block.  Reading for a tail block (n not a
 * multiple of B): it is zero-padded to B for the scale and for packing (the
 * padding's codes are the code of 0, or +1 for b = 1), the 1-bit mean
 * divides by the number of real elements, and only real elements get an
 * error-feedback value.  err_out may be NULL. */
static void quantize_stage(const float* v, int64_t n, const orc_params* p,
                           float* err_out, uint8_t* codes, uint16_t* scales)
{
    const int B = p->block, b = p->bits;
    const int64_t nb = orc_num_blocks(n, B);
    float* absv = new float[B];
    for (int64_t k = 0; k < nb; ++k) {
        int64_t first = k * B;
        int n_valid = (int)((n - first) < B ? (n - first) : B);
        for (int j = 0; j < B; ++j) absv[j] = (j < n_valid) ? fabsf(v[first + j]) : 0.0f;
        uint16_t sh = block_scale(absv, B, n_valid, b);
        scales[k] = sh;
        float s = orc_f16_to_f32(sh);
        for (int j = 0; j < B; ++j) {
            int64_t e = first + j;
            float val = (j < n_valid) ? v[e] : 0.0f;
            int32_t q = quantize_value(val, s, p, p->index_offset + (uint64_t)e);
            put_code(codes, e, b, offset_code(q, b));
            if (err_out && j < n_valid) {
                float d = s * (float)q;          /* separate roundings, no FMA */
                err_out[e] = val - d;
            }
        }
    }
    delete[] absv;
}

/* ------------------------------------------------------------------ */
/* Encoder                                                              */
/* ------------------------------------------------------------------ */

int orc_quantize_pack(const void* x, int32_t dtype, int64_t n, float* err,
                      const orc_params* p, uint8_t* codes, uint16_t* scales)
{
    if (!valid_params(p) || n < 0 || (dtype != 0 && dtype != 1)) return 1;
    if (n == 0) return 0;
    if (!x || !codes || !scales) return 1;
    if (p->hadamard && n % p->hadamard != 0) return 1;
    float* v = new float[n];
    for (int64_t i = 0; i < n; ++i)
        v[i] = (dtype == 0) ? ((const float*)x)[i] : orc_bf16_to_f32(((const uint16_t*)x)[i]);
    if (p->hadamard) orc_fwht(v, n, p->hadamard);  /* smoothing rotation of g */
    if (err)
        for (int64_t i = 0; i < n; ++i) v[i] = v[i] + err[i];   /* a1: EF add (fp32 RN) */
    quantize_stage(v, n, p, err, codes, scales);  /* a2-a6, e' written into err */
    delete[] v;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Decoder: unpack + dequantise W ranks, fixed rank-order fp32 sum,      */
/* optional stage-2 error feedback, requantise + repack.                */
/* ------------------------------------------------------------------ */

/* Reading of "local reduce": the SUM over ranks (averaging is the caller's),
 * accumulated in rank order starting from rank 0's value (not from 0.0f,
 * which would turn a -0 into +0): r = d_0; r = r + d_w for w = 1..W-1. */
int orc_unpack_dequant_reduce_requant(const uint8_t* const* codes_in,
                                      const uint16_t* const* scales_in,
                                      int32_t W, int64_t n, const orc_params* p_in,
                                      float* sum_out, float* err2,
                                      const orc_params* p_out,
                                      uint8_t* codes_out, uint16_t* scales_out)
{
    if (!valid_params(p_in) || W < 1 || n < 0) return 1;
    if (p_out && !valid_params(p_out)) return 1;
    /* the rank sum and the requantisation stay in the transformed domain */
    if (p_out && p_out->hadamard != p_in->hadamard) return 1;
    if (n == 0) return 0;
    if (!codes_in || !scales_in) return 1;
    for (int w = 0; w < W; ++w) if (!codes_in[w] || !scales_in[w]) return 1;
    if (p_out && (!codes_out || !scales_out)) return 1;

    const int bin = p_in->bits, Bin = p_in->block;
    float* r = new float[n];
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int w = 0; w < W; ++w) {
            float s = orc_f16_to_f32(scales_in[w][i / Bin]);
            int32_t q = code_to_q(get_code(codes_in[w], i, bin), bin);
            float d = s * (float)q;                  /* a8 dequantise */
            acc = (w == 0) ? d : acc + d;            /* a9 rank-ordered sum */
        }
        r[i] = acc;
        if (sum_out) sum_out[i] = acc;
    }
    if (p_out) {
        if (err2) for (int64_t i = 0; i < n; ++i) r[i] = r[i] + err2[i];   /* a10: v2 = r + e2 */
        quantize_stage(r, n, p_out, err2, codes_out, scales_out);      /* e2' = v2 - s2*q2 */
    }
    delete[] r;
    return 0;
}

/* Full-precision local reduce of the hierarchical all-reduce (bitscom README,
 * "Implemented Features": pipeline-A local reduce; "Hierarchical All-Reduce
 * Options": local_quantize=False keeps the local stage in full precision).
 * Reading: the W local ranks' values are summed in fp32 in rank order, rank
 * 0's value first: out = fl(...fl(x_0 + x_1)... + x_{W-1}); bf16 inputs are
 * widened exactly. */
int orc_sum_ranks(const void* const* x, int32_t dtype, int32_t W, int64_t n, float* out)
{
    if (!x || !out || W < 1 || n < 0 || (dtype != 0 && dtype != 1)) return 1;
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t w = 0; w < W; ++w) {
            float v = (dtype == 0) ? ((const float*)x[w])[i] : orc_bf16_to_f32(((const uint16_t*)x[w])[i]);
            s = (w == 0) ? v : s + v;
        }
        out[i] = s;
    }
    return 0;
}

/* The all-gather side of the low-bit all-reduce: after the all-gather every
 * rank holds the requantised chunks of all ranks (bitscom README,
 * "Implemented Features": all-to-all -> local reduce -> all-gather) and
 * decodes them into its gradient.  The reduce is a SUM; averaging is the
 * caller's multiplier (reading: mul = 1/W gives the mean). */
int orc_unpack_dequant(const uint8_t* codes, const uint16_t* scales, int64_t n,
                       const orc_params* p, float mul, int32_t out_dtype, void* out)
{
    if (!valid_params(p) || n < 0 || (out_dtype != 0 && out_dtype != 1)) return 1;
    if (n == 0) return 0;
    if (!codes || !scales || !out) return 1;
    const int H = p->hadamard;
    if (H && n % H != 0) return 1;
    float* d = new float[n];
    for (int64_t i = 0; i < n; ++i) {
        float s = orc_f16_to_f32(scales[i / p->block]);
        int32_t q = code_to_q(get_code(codes, i, p->bits), p->bits);
        d[i] = s * (float)q;
    }
    if (H) {   /* inverse rotation: the same transform, then 1/H (exact) */
        orc_fwht(d, n, H);
        float inv = ldexpf(1.0f, -(int)log2((double)H));
        for (int64_t i = 0; i < n; ++i) d[i] = d[i] * inv;
    }
    for (int64_t i = 0; i < n; ++i) {
        float y = d[i] * mul;
        if (out_dtype == 0) ((float*)out)[i] = y;
        else ((uint16_t*)out)[i] = orc_f32_to_bf16(y);
    }
    delete[] d;
    return 0;
}

/* SDP4Bit README, "Weight Quantization Arguments" (--quantized-weights,
 * --weight-quantization-bits, --wq-group-size) and its overview ("quantization
 * on weight differences").  Reading: the difference is taken against the
 * reference copy every rank already holds (the last broadcast weights), the
 * reference advances by the dequantised difference on every rank -- the
 * sender included, so all copies stay bit-identical -- and the quantisation
 * residual stays in w - ref for the next step.  No Hadamard rotation here. */
int orc_qwd_encode(const void* w, int32_t dtype, int64_t n, float* ref, const orc_params* p,
                   uint8_t* codes, uint16_t* scales)
{
    if (!valid_params(p) || p->hadamard || n < 0 || (dtype != 0 && dtype != 1)) return 1;
    if (n == 0) return 0;
    if (!w || !ref || !codes || !scales) return 1;
    float* d = new float[n];
    for (int64_t i = 0; i < n; ++i) {
        float wi = (dtype == 0) ? ((const float*)w)[i] : orc_bf16_to_f32(((const uint16_t*)w)[i]);
        d[i] = wi - ref[i];
    }
    quantize_stage(d, n, p, NULL, codes, scales);
    delete[] d;
    return orc_qwd_apply(codes, scales, n, p, ref, NULL, 0);
}

int orc_qwd_apply(const uint8_t* codes, const uint16_t* scales, int64_t n, const orc_params* p,
                  float* ref, void* w_out, int32_t w_dtype)
{
    if (!valid_params(p) || p->hadamard || n < 0 || (w_dtype != 0 && w_dtype != 1)) return 1;
    if (n == 0) return 0;
    if (!codes || !scales || !ref) return 1;
    for (int64_t i = 0; i < n; ++i) {
        float s = orc_f16_to_f32(scales[i / p->block]);
        int32_t q = code_to_q(get_code(codes, i, p->bits), p->bits);
        ref[i] = ref[i] + s * (float)q;
        if (w_out) {
            if (w_dtype == 0) ((float*)w_out)[i] = ref[i];
            else ((uint16_t*)w_out)[i] = orc_f32_to_bf16(ref[i]);
        }
    }
    return 0;
}

int orc_roundtrip(const void* x, int32_t dtype, int64_t n, float* err,
                  const orc_params* p, uint8_t* codes, uint16_t* scales, float* deq_out)
{
    int rc = orc_quantize_pack(x, dtype, n, err, p, codes, scales);
    if (rc || n == 0) return rc;
    return orc_unpack_dequant(codes, scales, n, p, 1.0f, 0, deq_out);
}
