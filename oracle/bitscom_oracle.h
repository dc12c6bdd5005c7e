/*
 * bitscom_oracle.h -- plain, slow, single-threaded CPU oracle of the low-bit
 * gradient codec.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the CPU-baseline leg of the benchmark may load it; the library's product
 * path never does.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (steps in the order they run):
 *   encoder  : v = g (+ e)  ->  per-block scale s (fp16)  ->  codes q  ->
 *              e' = v - s*q  ->  offset-binary codes packed LSB-first.
 *   decoder  : unpack W ranks' codes -> d_w = s_w*q_w -> rank-ordered fp32
 *              sum -> (+ e2) -> requantise + repack with stage-2 parameters.
 * The feature list comes from the bitscom README (Aerithy/bitscom),
 * "Implemented Features": bitwidths 1/2/4/8/12/16, tensor quantize /
 * dequantize, bit-packing, stochastic rounding, blockwise quantisation with
 * per-block FP16 scales, the all-to-all -> local reduce -> all-gather
 * all-reduce, first-stage error feedback and stage2_error_feedback.
 *
 * All integers are little-endian; codes are produced as a byte stream.
 * Every function returns 0 on success and a nonzero value on a bad argument.
 *
 * Parity status: every function here is pinned by tests against values fixed
 * by the pages and the mathematics (hand-worked blocks, exhaustive format
 * conversions, cuRAND's host Philox, closed-form bounds, numpy packbits,
 * scipy's Hadamard matrix).  Two readings have no support in the pages: the
 * zero-padded tail block (n mod B != 0) and stochastic rounding at 1 bit
 * (taken as plain sign); their implementation is pinned to the reading
 * (hand-worked tail blocks, tail == zero-padded block, 1-bit SR == RTN), the
 * reading itself is not.
 */
#ifndef BITSCOM_ORACLE_H
#define BITSCOM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One quantisation stage's parameters (the oracle's own definition). */
typedef struct {
    int32_t  bits;           /* 1, 2, 4, 8, 12 or 16                      */
    int32_t  block;          /* power of two, >= 8                        */
    int32_t  rounding;       /* 0 = round half to even, 1 = stochastic    */
    uint32_t philox_stream;  /* third Philox counter word                 */
    uint64_t seed;           /* Philox key                                */
    uint64_t index_offset;   /* global element index of element 0         */
    int32_t  hadamard;       /* 0, or the Walsh-Hadamard transform block H */
    int32_t  reserved;
} orc_params;

/* IEEE-754 conversions written from the format definitions. */
uint16_t orc_f32_to_f16(float x);            /* round to nearest even     */
float    orc_f16_to_f32(uint16_t h);
float    orc_bf16_to_f32(uint16_t b);
void     orc_f32_to_f16_many(const float* x, uint16_t* out, int64_t n);

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* The 32-bit random word the codec draws for global element index i. */
uint32_t orc_random_word(uint64_t seed, uint32_t stream, uint64_t i);
/* The words of elements i0 .. i0+n-1, one orc_random_word call each (a test helper). */
void orc_random_words(uint64_t seed, uint32_t stream, uint64_t i0, int64_t n, uint32_t* out);

/* Encoder.  dtype 0 = fp32, 1 = bf16 (raw uint16 bits).  err may be NULL
 * (no error feedback).  codes receives packed_bytes(n) bytes, scales
 * num_blocks(n) fp16 bit patterns. */
int orc_quantize_pack(const void* x, int32_t dtype, int64_t n, float* err,
                      const orc_params* p, uint8_t* codes, uint16_t* scales);

/* Decoder over W ranks' codes of one chunk of n elements.  sum_out and err2
 * may be NULL; p_out NULL means no requantisation. */
int orc_unpack_dequant_reduce_requant(const uint8_t* const* codes_in,
                                      const uint16_t* const* scales_in,
                                      int32_t W, int64_t n, const orc_params* p_in,
                                      float* sum_out, float* err2,
                                      const orc_params* p_out,
                                      uint8_t* codes_out, uint16_t* scales_out);

/* Encoder then all-gather-side decode with mul = 1: deq_out = s*q per element
 * (inverse-transformed when p->hadamard is set). */
int orc_roundtrip(const void* x, int32_t dtype, int64_t n, float* err,
                  const orc_params* p, uint8_t* codes, uint16_t* scales, float* deq_out);

/* All-gather-side decode: out[i] = fl(fl(s*q) * mul) for i < n, written as
 * fp32 (out_dtype 0) or bf16 bits (out_dtype 1, round to nearest even). */
int orc_unpack_dequant(const uint8_t* codes, const uint16_t* scales, int64_t n,
                       const orc_params* p, float mul, int32_t out_dtype, void* out);
uint16_t orc_f32_to_bf16(float x);

/* Full-precision local reduce: out[i] = fl(...fl(x_0[i] + x_1[i])... +
 * x_{W-1}[i]) in fp32, rank order, rank 0's value first (dtype 0 = fp32,
 * 1 = bf16 bits). */
int orc_sum_ranks(const void* const* x, int32_t dtype, int32_t W, int64_t n, float* out);

/* Weight-difference quantisation for the sharded weight all-gather.
 * Sender: d = fl(w - ref) quantised (codes, scales); ref = fl(ref + fl(s*q)).
 * Receiver (every rank, on the gathered codes): ref = fl(ref + fl(s*q)), and
 * optionally w_out = ref as fp32 (w_dtype 0) or bf16 bits (1). */
int orc_qwd_encode(const void* w, int32_t dtype, int64_t n, float* ref, const orc_params* p,
                   uint8_t* codes, uint16_t* scales);
int orc_qwd_apply(const uint8_t* codes, const uint16_t* scales, int64_t n, const orc_params* p,
                  float* ref, void* w_out, int32_t w_dtype);

/* Unnormalised fast Walsh-Hadamard transform of every H-element block of
 * x[0:n) in place (n a multiple of H). */
int orc_fwht(float* x, int64_t n, int32_t H);

/* Sizes. */
int64_t orc_num_blocks(int64_t n, int32_t block);
int64_t orc_packed_bytes(int64_t n, int32_t bits, int32_t block);

#ifdef __cplusplus
}
#endif
#endif
