/*
 * bitscom.h -- C ABI of the GB300 low-bit gradient codec.
 *
 * The data-parallel hot path of a low-bit all-reduce: blockwise quantise +
 * bit-pack + error feedback on every rank (encoder), then, between the
 * all-to-all and the all-gather, unpack + dequantise + fixed-order reduce +
 * requantise + repack of each rank's chunk (decoder).  Feature set from the
 * bitscom README (Aerithy/bitscom), "Implemented Features": bitwidths
 * 1/2/4/8/12/16, quantize/dequantize, bit-packing, stochastic rounding,
 * blockwise quantization with per-block FP16 scales, the low-bit all-reduce
 * pipeline (all-to-all -> local reduce -> all-gather), first-stage error
 * feedback; "Backend Registration Options": stage2_error_feedback.  The
 * split of an all-reduce into a reduce-scatter and an all-gather is the
 * subject of the DeAR README; 25 MB tensor-fusion buckets are the default
 * of both the ACP-SGD and DeAR READMEs.
 *
 * Arithmetic (the pages leave it open; this library fixes it):
 *   Qmax = 2^(b-1) - 1.
 *   b >= 2: s = fp16_rne(min(absmax_fp32 / Qmax, 65504)), division correctly
 *           rounded in fp32; q = clamp(rint_half_even(v / s), -Qmax, Qmax);
 *           s == 0 gives q = 0.
 *   b == 1: s = fp16_rne(min(mean|v|, 65504)) with the block sum taken as a
 *           balanced binary tree over contiguous halves of the zero-padded
 *           block and divided by the number of real elements; q = +1 if
 *           v >= 0 (both zeros) else -1; the rounding mode is ignored.
 *   Stochastic rounding: t = v/s, f = floor(t), p = t - f (exact), u =
 *           (r mod 2^23) * 2^-23 with r = word (i mod 4) of Philox4x32-10
 *           (counter = (i/4 low, i/4 high, philox_stream, 0), key = (seed low,
 *           seed high)), i = index_offset + element index; q = clamp(f +
 *           [u < p], -Qmax, Qmax).
 *   Codes: offset binary u = q + 2^(b-1) (b >= 2) or (q + 1)/2 (b = 1),
 *           packed LSB-first into a little-endian byte stream; block k's
 *           codes start at byte k*B*b/8.  A tail block is zero-padded.
 *   Error feedback: v = fl(g + e); e' = fl(v - fl(s*q)) (no fused multiply-add).
 *   Reduce: r = d_0, r = fl(r + d_w) for w = 1..W-1 (rank order, fp32), with
 *           d_w = fl(s_w * q_w); stage 2 adds e2: v2 = fl(r + e2).
 *   Hadamard smoothing (SDP4Bit README, "--hadamard-transform"; optional):
 *           the encoder rotates every H-element block of g by the unnormalised
 *           Sylvester Walsh-Hadamard transform (stage h = 1, 2, 4, ...: x_i,
 *           x_{i+h} -> x_i + x_{i+h}, x_i - x_{i+h} in fp32) before adding e;
 *           error feedback, the rank sum and the requantisation stay in the
 *           rotated domain; bitscom_unpack_dequant applies the inverse (the
 *           same transform, then 1/H).
 *
 * Memory: the caller allocates and owns every buffer (device memory unless
 * stated) and the CUDA stream.  Calls are asynchronous on the given stream
 * (NULL = legacy default stream); a call enqueues kernels and returns.  The
 * entry points above the scheduler section allocate nothing; except for
 * bitscom_roundtrip_noalloc (its own rules below) they keep no state between
 * calls and may be called from several host threads.
 *
 * Errors: arguments are checked on the host before anything is enqueued:
 *   BITSCOM_EINVAL       bits not in {1,2,4,8,12,16}, block not a power of two
 *                        in [8, 4096], rounding not 0/1, n < 0, a required
 *                        pointer NULL while n > 0, W outside [1, 64].
 *   BITSCOM_EALIGN       a pointer below its required alignment (stated per
 *                        argument).
 *   BITSCOM_EUNSUPPORTED a (bits_in, bits_out) pair the decoder has no kernel for.
 *   BITSCOM_ECUDA        a CUDA runtime error while enqueueing.
 * Faults inside a kernel surface at the caller's next synchronisation.
 * n == 0 enqueues nothing and returns BITSCOM_OK.
 */
#ifndef BITSCOM_H
#define BITSCOM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BITSCOM_OK = 0,
    BITSCOM_EINVAL = 1,
    BITSCOM_EALIGN = 2,
    BITSCOM_EUNSUPPORTED = 3,
    BITSCOM_ECUDA = 4,
    BITSCOM_ETIMEOUT = 5
} bitscom_status;

typedef enum { BITSCOM_F32 = 0, BITSCOM_BF16 = 1 } bitscom_dtype;
typedef enum { BITSCOM_RTN = 0, BITSCOM_SR = 1 } bitscom_rounding;

/* Parameters of one quantisation stage (the options of bitscom.init():
 * bitwidth, block_size, stochastic rounding). */
typedef struct {
    int32_t  bits;           /* 1, 2, 4, 8, 12, 16                                  */
    int32_t  block;          /* B: power of two, 8..4096                            */
    int32_t  rounding;       /* bitscom_rounding; ignored for bits == 1             */
    uint32_t philox_stream;  /* Philox counter word 2 (0 = stage 1, 1 = stage 2)    */
    uint64_t seed;           /* Philox key                                          */
    uint64_t index_offset;   /* global element index of element 0 of this call      */
    int32_t  hadamard;       /* 0, or H: rotate every H-element block by the        */
                             /* Walsh-Hadamard transform (H a power of two in        */
                             /* [8, 256] dividing block; bits 2, 4 or 8; n a         */
                             /* multiple of H).  Every stage of one all-reduce uses  */
                             /* the same H.                                          */
    int32_t  reserved;       /* must be 0                                           */
} bitscom_qparams;

/* Number of blocks ceil(n / block). */
int64_t bitscom_num_blocks(int64_t n, int32_t block);
/* Bytes of packed codes for n elements: num_blocks * block * bits / 8. */
int64_t bitscom_packed_bytes(int64_t n, int32_t bits, int32_t block);
/* Static English text of a status code. */
const char* bitscom_status_string(bitscom_status s);
/* Text of the last CUDA error this thread saw inside the library ("" if none). */
const char* bitscom_last_cuda_error(void);

/*
 * Encoder: per-block absmax (mean for b = 1) + scale + quantise + pack, with
 * optional first-stage error feedback.  bitscom README, "Implemented
 * Features" (blockwise quantization with per-block FP16 scales; error
 * feedback in first-stage quantization).
 *   x          [n] gradients, fp32 (32-byte aligned) or bf16 (16-byte aligned).
 *   err        [n] fp32 error buffer, in/out (32-byte aligned); NULL = no error
 *              feedback.  Read as e, overwritten with e'.
 *   p          stage parameters (host pointer).
 *   codes_out  packed_bytes(n) bytes; aligned to the per-thread store width:
 *              1 (b=1), 2 (b=2), 4 (b=4, 12), 8 (b=8), 16 (b=16) bytes.
 *   scales_out [num_blocks] fp16 bit patterns (2-byte aligned).
 * Buffers must not overlap.  Performance note: without error feedback a
 * codes_out aligned to twice the store width (and blocks of >= 16) lets the
 * encoder handle 16 elements per thread; with stochastic rounding, b >= 2,
 * blocks of 32 .. 4096 and codes_out 16-byte aligned (8 at b = 2) it handles
 * 32, which measured 1.2x faster (fp32, 4-bit, block 128).  The results are
 * the same bits on every path.
 */
bitscom_status bitscom_quantize_pack(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                     const bitscom_qparams* p, void* codes_out,
                                     uint16_t* scales_out, void* cuda_stream);

/*
 * Decoder of one chunk between the all-to-all and the all-gather: for each
 * of n elements, unpack and dequantise the W ranks' codes (d_w = s_w * q_w),
 * sum them in rank order in fp32, optionally write the sum, optionally add
 * the stage-2 error e2, requantise with p_out and repack, writing e2'.
 * bitscom README, "Implemented Features" (all-to-all -> local reduce ->
 * all-gather) and "Backend Registration Options" (stage2_error_feedback /
 * ef21_plus: error feedback on the reduced-shard quantisation).
 *   codes_in   host array of W device pointers to each rank's packed codes of
 *              this chunk (block-aligned chunk start), aligned as codes_out of
 *              the encoder for p_in->bits.
 *   scales_in  host array of W device pointers to fp16 scales (2-byte aligned).
 *   p_in       bits/block of the incoming codes (rounding/seed unused).
 *   sum_out    [n] fp32 rank-ordered sum (32-byte aligned); NULL = not written.
 *   err2       [n] fp32 stage-2 error, in/out (32-byte aligned); NULL = none.
 *              Requires p_out.
 *   p_out      stage-2 parameters; NULL = no requantisation (codes_out and
 *              scales_out are then ignored).
 *   codes_out, scales_out   as in the encoder, for p_out.
 * The decoder has kernels for bits_out in {none, bits_in} and for the
 * two-level pair (8 -> 4); other pairs return BITSCOM_EUNSUPPORTED.
 * Performance note: for W = 8 and 4 -> 4 bits, 8-byte aligned codes_in and
 * codes_out (and blocks of >= 16) let the decoder handle 16 elements per
 * thread, and so do 8-byte aligned codes_in for W = 8 4-bit codes decoded into
 * sum_out alone (no p_out, no err2); W = 1 without p_out runs the all-gather-
 * side decode with mul = 1.  The results are the same bits on every path.
 */
bitscom_status bitscom_unpack_dequant_reduce_requant(
    const void* const* codes_in, const uint16_t* const* scales_in, int32_t W, int64_t n,
    const bitscom_qparams* p_in, float* sum_out, float* err2, const bitscom_qparams* p_out,
    void* codes_out, uint16_t* scales_out, void* cuda_stream);

/*
 * All-gather-side decode: after the all-gather of the low-bit all-reduce every
 * rank holds all ranks' requantised chunks (bitscom README, "Implemented
 * Features": all-to-all -> local reduce -> all-gather) and decodes them into
 * its gradient: out[i] = fl(fl(s*q) * mul), written as fp32 (out 32-byte
 * aligned) or bf16 (round to nearest even, out 16-byte aligned).  The reduce
 * is a SUM; mul = 1/W turns it into the mean.
 *   codes, scales   one stream of packed codes / fp16 scales of n elements for
 *                   p (alignment as the encoder's outputs).
 * Performance note: with blocks of >= 16, no rotation, codes aligned to twice
 * the encoder's store width and out 32-byte aligned, the decode handles 16
 * elements per thread; with a rotation (p->hadamard != 0), blocks of >= 32,
 * codes 8-byte (b = 2) or 16-byte (b = 4, 8) aligned and out 32-byte aligned,
 * it handles 32 and keeps up to five stages of the transform in registers
 * (H = 128 into bf16: 1.8x the 8-element kernel).  The results are the same
 * bits on every path.
 */
bitscom_status bitscom_unpack_dequant(const void* codes, const uint16_t* scales, int64_t n,
                                      const bitscom_qparams* p, float mul, bitscom_dtype out_dt,
                                      void* out, void* cuda_stream);

/*
 * Rank-ordered fp32 sum of W full-precision arrays: the local reduce of the
 * hierarchical all-reduce when local communication is not quantised (bitscom
 * README, "Implemented Features": hierarchical pipeline-A, local reduce ->
 * inter low-bit all-reduce -> local broadcast; "Hierarchical All-Reduce
 * Options": local_quantize=False, local full precision).
 *   out[i] = fl(...fl(fl(x_0[i]) + x_1[i]) ... + x_{W-1}[i]): rank 0 sets the
 *   sum (so -0 stays -0), the others are added in rank order in fp32 -- a
 *   fixed order, unlike a collective's reduction.
 *   x    host array of W device pointers (W in [1, 64]) to n elements each,
 *        fp32 (32-byte aligned) or bf16 (16-byte aligned, converted exactly).
 *   out  [n] fp32 (32-byte aligned); may not overlap any x[w].
 */
bitscom_status bitscom_sum_ranks(const void* const* x, bitscom_dtype dt, int32_t W, int64_t n, float* out,
                                 void* cuda_stream);

/*
 * Weight-difference quantisation for the sharded weight all-gather (SDP4Bit
 * README, "Weight Quantization Arguments": --quantized-weights,
 * --weight-quantization-bits 4, --wq-group-size 2048; "quantization on weight
 * differences").  The shard owner quantises d = fl(w - ref) against the
 * reference copy every rank holds and advances its own copy:
 * ref = fl(ref + fl(s*q)); every rank then applies the all-gathered codes to
 * its copy with bitscom_qwd_apply, so all copies stay bit-identical and the
 * residual w - ref carries into the next step.  Bits 2, 4, 8; no Hadamard.
 *   w          [n] weights, fp32 (32-byte aligned) or bf16 (16-byte aligned).
 *   ref        [n] fp32 reference, in/out (32-byte aligned).
 *   codes_out, scales_out   as in bitscom_quantize_pack.
 */
bitscom_status bitscom_qwd_encode(const void* w, bitscom_dtype dt, int64_t n, float* ref,
                                  const bitscom_qparams* p, void* codes_out, uint16_t* scales_out,
                                  void* cuda_stream);
/* Receiver side: ref = fl(ref + fl(s*q)) for n elements of gathered codes;
 * w_out (NULL = none) receives the new weights as fp32 or bf16 (w_dt).
 * Performance note: with blocks of >= 16, codes aligned to twice the encoder's
 * store width and w_out 32-byte aligned (or NULL), the apply handles 16
 * elements per thread; the results are the same bits on every path. */
bitscom_status bitscom_qwd_apply(const void* codes, const uint16_t* scales, int64_t n,
                                 const bitscom_qparams* p, float* ref, void* w_out,
                                 bitscom_dtype w_dt, void* cuda_stream);

/*
 * Quantise then dequantise (the simulate_quantization mode of "Implemented
 * Features"): the codes and scales go to caller scratch codes_tmp /
 * scales_tmp and fl(s*q) to deq_out.  Without error feedback and rotation the
 * encoder writes all three in one pass; otherwise the encoder runs, then the
 * single-rank decoder.  deq_out may alias x when dt == F32.
 */
bitscom_status bitscom_roundtrip(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                 const bitscom_qparams* p, void* codes_tmp,
                                 uint16_t* scales_tmp, float* deq_out, void* cuda_stream);

/*
 * Allocation-free variant of bitscom_roundtrip (the pages have no counterpart;
 * this is a library convenience).  For callers that cannot allocate device
 * memory where they quantise -- e.g. a gradient hook that only holds the
 * gradient buffer and must not call the CUDA allocator, which can synchronise
 * the device and compete with a framework's caching allocator.  The codes and
 * scales live in a fixed device array of this library (8 MiB of codes + 1 MiB
 * of scales per device); the caller still passes x, err and deq_out as in
 * bitscom_roundtrip, and the results are identical to it.
 *   - n must not exceed bitscom_roundtrip_noalloc_max_elements(bits, block)
 *     (at least 4,194,304 for every bits/block; 16,777,216 for 4-bit, block
 *     128); larger n returns BITSCOM_EINVAL and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  With CUDA's default
 *     lazy module loading that lookup is what reserves the 9 MiB on the
 *     device, and it may synchronise the device; it fails with BITSCOM_ECUDA
 *     if the device has no 9 MiB left.  So make that first call at set-up
 *     time, while memory is still free and before any stream capture on the
 *     device.  The array then stays until the process exits.
 *   - The address is kept per device number: after cudaDeviceReset (which
 *     destroys the array) calls on that device are not supported.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing in it needs clearing: every code and scale is written
 *     before it is read).  Calls whose kernels overlap on the GPU race on it.
 *   - Allocates nothing: no cudaMalloc / cudaFree or allocating library call.
 */
bitscom_status bitscom_roundtrip_noalloc(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                         const bitscom_qparams* p, float* deq_out,
                                         void* cuda_stream);
/* Largest n bitscom_roundtrip_noalloc accepts for these parameters (-1 if the
 * parameters are invalid). */
int64_t bitscom_roundtrip_noalloc_max_elements(int32_t bits, int32_t block);

/* ------------------------------------------------------------------------
 * Bucket scheduler: splits a flat gradient into fusion buckets (25 MB by
 * default in the ACP-SGD and DeAR READMEs) and runs them round-robin on its
 * own CUDA streams (bitscom README, "Implemented Features": dual-stream
 * scheduling).  The scheduler owns its streams and events (no device memory).
 * Every call is ordered after earlier work on cuda_stream, and later work on
 * cuda_stream is ordered after all of the call's buckets.  Buckets are
 * block-aligned and each bucket's Philox indices are its global element
 * indices, so results are bit-identical to one unbucketed call.  One
 * scheduler must not be used from two host threads at once.
 * ------------------------------------------------------------------------ */
typedef struct bitscom_sched bitscom_sched;

/* n_streams in [1, 8]; bucket_bytes <= 0 means one bucket per call. */
bitscom_status bitscom_sched_create(int32_t n_streams, int64_t bucket_bytes, bitscom_sched** out);
bitscom_status bitscom_sched_destroy(bitscom_sched* s);

/* Host-only planner: bucket k covers elements [starts[k], starts[k+1]) of n
 * elements of elem_bytes each; buckets hold floor(bucket_bytes / elem_bytes)
 * elements rounded down to a multiple of max(block, 128) (at least one such
 * unit).  Writes up to cap+1 entries and returns the number of buckets, or -1
 * on bad arguments.  starts may be NULL to only count. */
int64_t bitscom_sched_plan(int64_t n, int32_t elem_bytes, int32_t block, int64_t bucket_bytes,
                           int64_t* starts, int64_t cap);

/* Bucketed encoder; arguments as bitscom_quantize_pack. */
bitscom_status bitscom_sched_quantize_pack(bitscom_sched* s, const void* x, bitscom_dtype dt,
                                           int64_t n, float* err, const bitscom_qparams* p,
                                           void* codes_out, uint16_t* scales_out,
                                           void* cuda_stream);

/*
 * Simulated W-rank low-bit all-reduce on one GPU: the W ranks' gradients are
 * W device arrays.  Per bucket: each rank's encoder (p1[w], error buffer
 * err[w]) writes codes[w] / scales[w]; the bucket's blocks are split into W
 * chunks of ceil(nb/W) blocks (the all-to-all is pointer arithmetic) and each
 * chunk's decoder sums the W ranks in rank order, adds err2 (the chunk
 * owner's stage-2 error) and requantises with p2 into codes_out / scales_out
 * at the chunk's global position (what the all-gather would distribute).
 *   x[W], err[W] (NULL entries or err == NULL: no first-stage feedback),
 *   p1[W] (host array), codes[W], scales[W]: per-rank buffers of n elements.
 *   p2: stage-2 parameters (NULL: no requantisation; sum_out must then be set).
 *   err2 [n] (NULL: no stage-2 feedback); codes_out / scales_out for p2;
 *   sum_out [n] fp32 rank-ordered sum, or NULL.
 */
bitscom_status bitscom_sched_allreduce(bitscom_sched* s, int32_t W, const void* const* x,
                                       bitscom_dtype dt, int64_t n, float* const* err,
                                       const bitscom_qparams* p1, void* const* codes,
                                       uint16_t* const* scales, const bitscom_qparams* p2,
                                       float* err2, void* codes_out, uint16_t* scales_out,
                                       float* sum_out, void* cuda_stream);

/* Host wait for all work enqueued on cuda_stream, polling with a deadline:
 * BITSCOM_OK, BITSCOM_ETIMEOUT (work still running after timeout_s seconds)
 * or BITSCOM_ECUDA (the stream reported an error). */
bitscom_status bitscom_sched_wait(bitscom_sched* s, void* cuda_stream, double timeout_s);

#ifdef __cplusplus
}
#endif
#endif /* BITSCOM_H */
