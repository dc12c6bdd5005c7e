// decode_impl.cuh -- fused decoder kernel for one chunk between the all-to-all and
// the all-gather of a low-bit all-reduce: unpack + dequantise the W ranks'
// codes, sum them in rank order in fp32, optionally add the stage-2 error,
// requantise + repack (bitscom README, "Implemented Features": all-to-all ->
// local reduce -> all-gather; "Backend Registration Options":
// stage2_error_feedback).  Every byte of the W inputs is read once and every
// output byte written once; the rank sum never leaves registers.
#pragma once

#include "codec.cuh"
#include "launch.h"

namespace bitscom {

// One rank's contribution to the 8 running sums: acc = fl(acc + fl(s*q)), or
// acc = fl(s*q) for the first rank.  For b in {2, 4, 8} the fp16 scale and
// fp16 levels feed a mixed-precision fma (s*q exact, one rounding); for b = 1
// and 12 the fp32 fma is exact for the same reason; at b = 16 s*q may need 27
// bits, so the multiply and the add round separately.
template <int BITS>
__device__ __forceinline__ void accumulate_rank(const Packed<BITS>& c, unsigned short sbits, bool first,
                                                float (&acc)[8])
{
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
        uint32_t h[4];
        level_pairs<BITS>(c, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int jl = pair_lo<BITS>(i), jh = pair_hi<BITS>(i);
            const unsigned short ql = (unsigned short)(h[i] & 0xFFFFu), qh = (unsigned short)(h[i] >> 16);
            acc[jl] = fma_f16(sbits, ql, first ? -0.0f : acc[jl]);
            acc[jh] = fma_f16(sbits, qh, first ? -0.0f : acc[jh]);
        }
    } else {
        const float s = __half2float(__ushort_as_half(sbits));
        float l[8];
        levels8<BITS>(c, l);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (first) {
                acc[j] = __fmul_rn(s, l[j]);
            } else if constexpr (BITS <= 12) {
                acc[j] = __fmaf_rn(s, l[j], acc[j]);
            } else {
                acc[j] = __fadd_rn(acc[j], __fmul_rn(s, l[j]));
            }
        }
    }
}

// The first (up to) 8 ranks' codes and fp16 scales of one thread's piece.
template <int BIN>
struct RowCodes {
    Packed<BIN> c[8];
    unsigned short s[8];
};

template <int BIN, int KW>
__device__ __forceinline__ void load_row_codes(const DecArgs& a, int64_t row, RowCodes<BIN>& r)
{
    const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
    if (e0 >= a.n) return;
    const int64_t piece = e0 >> 3, blk_in = e0 >> a.log2Bin;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (KW == 8 || k < a.W) {
            r.c[k] = load_codes<BIN>(a.codes[k], piece);
            r.s[k] = __ldg(a.scales[k] + blk_in);
        }
    }
}

// The rest of a row once its rank sum is in registers: the optional fp32 sum,
// then stage-2 error feedback, block statistic, requantisation, packing and
// the new stage-2 error.  `e2` holds the row's incoming stage-2 error (read
// only when a.err2 is set); `red` is this row's half of the team exchange.
template <int BOUT, bool SR>
__device__ __forceinline__ void finish_row(const DecArgs& a, int64_t e0, int valid, const float (&acc)[8],
                                           const float (&e2)[8], float* red)
{
    const int64_t n = a.n;
    const int64_t piece = e0 >> 3;
    if (a.sum_out != nullptr) {
        if (valid == 8) {
            st8_f32(a.sum_out + e0, acc);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) if (j < valid) a.sum_out[e0 + j] = acc[j];
        }
    }

    if constexpr (BOUT != 0) {
        const Team team = make_team(a.log2Bout);
        float v[8];
        if (valid == 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = a.err2 != nullptr ? __fadd_rn(acc[j], e2[j]) : acc[j];
        } else if (a.err2 != nullptr) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (j < valid) ? __fadd_rn(acc[j], e2[j]) : 0.0f;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (j < valid) ? acc[j] : 0.0f;
        }

        float stat;
        if constexpr (BOUT == 1) {
            stat = __fadd_rn(__fadd_rn(__fadd_rn(fabsf(v[0]), fabsf(v[1])), __fadd_rn(fabsf(v[2]), fabsf(v[3]))),
                             __fadd_rn(__fadd_rn(fabsf(v[4]), fabsf(v[5])), __fadd_rn(fabsf(v[6]), fabsf(v[7]))));
        } else {
            stat = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                         fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
        }
        stat = team_reduce<BOUT == 1>(stat, team, red);

        const int64_t blk = e0 >> a.log2Bout;
        int n_valid = 1 << a.log2Bout;
        if constexpr (BOUT == 1) {
            const int64_t left = n - (blk << a.log2Bout);
            if (left < n_valid) n_valid = left > 0 ? (int)left : 1;
        }
        const __half sh = block_scale<BOUT>(stat, n_valid);
        const float s2 = __half2float(sh);

        uint32_t rw[8];
        if constexpr (SR && BOUT > 1) {
            random_words8(a.index_offset + (uint64_t)e0, a.keys, (uint32_t)(a.index_offset & 3u), rw);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) rw[j] = 0u;
        }
        Packed<BOUT> c;
        float q[8];
        quantize8<BOUT, (SR && BOUT > 1)>(v, s2, scale_reciprocal(s2), rw, c, q);

        if (e0 < (a.nb_out << a.log2Bout)) store_codes<BOUT>(a.codes_out, piece, c);
        if (team.lane == 0 && blk < a.nb_out) a.scales_out[blk] = __half_as_ushort(sh);

        if (a.err2 != nullptr) {
            float e[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = feedback<BOUT>(v[j], s2, q[j]);
            if (valid == 8) {
                st8_f32(a.err2 + e0, e);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) a.err2[e0 + j] = e[j];
            }
        }
    }
}

// BOUT == 0: no requantisation (sum only).  MANY: W may exceed 8 (ranks 8..W-1
// are taken in groups of 8 inside the row; the kernel gets a larger register
// budget).  The row loop is software-pipelined: the next row's codes and
// scales of ranks 0..7 are loaded after the current row's ranks are summed,
// so they are in flight while it is requantised; the current row's stage-2
// error is loaded right after them (issued before the rank sum instead, it
// held 8 registers through it and measured 12 % slower: 0.364 vs 0.322 ms
// for a W = 8 chunk of 1.625e8 outputs).
// KW == 8: exactly eight ranks, known at compile time (the all-reduce of one
// eight-GPU node); KW == 0: the rank count is read from the arguments.
template <int BIN, int BOUT, bool SR, bool MANY, int KW>
__global__ void __launch_bounds__(kThreads, (MANY || BIN >= 12 || BOUT >= 12 || (SR && BIN >= 8)) ? 1 : 2)
decode_kernel(const DecArgs a)
{
    constexpr int kGroup = 8;   // ranks whose loads are issued together
    __shared__ float red[2][kWarps];
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    const int W = KW == 8 ? 8 : a.W;
    int parity = 0;

    RowCodes<BIN> cur;
    if ((int64_t)blockIdx.x < rows) load_row_codes<BIN, KW>(a, blockIdx.x, cur);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t piece = e0 >> 3;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        const int64_t blk_in = e0 >> a.log2Bin;

        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        if (valid > 0) {
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                if (k < W) accumulate_rank<BIN>(cur.c[k], cur.s[k], k == 0, acc);
            }
            if constexpr (MANY) {
#pragma unroll 1
                for (int w0 = kGroup; w0 < W; w0 += kGroup) {
                    Packed<BIN> c[kGroup];
                    unsigned short sh[kGroup];
#pragma unroll
                    for (int k = 0; k < kGroup; ++k) {
                        if (w0 + k < W) {
                            c[k] = load_codes<BIN>(a.codes[w0 + k], piece);
                            sh[k] = __ldg(a.scales[w0 + k] + blk_in);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kGroup; ++k) {
                        if (w0 + k < W) accumulate_rank<BIN>(c[k], sh[k], false, acc);
                    }
                }
            }
        }
        // prefetch: the next row's codes overlap this row's requantisation
        if (row + gridDim.x < rows) load_row_codes<BIN, KW>(a, row + gridDim.x, cur);
        // stage-2 error of this row, after the next row's codes are in flight
        float e2[8];
        if constexpr (BOUT != 0) {
            if (a.err2 != nullptr) {
                if (valid == 8) {
                    ld8_f32(a.err2 + e0, e2);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) e2[j] = (j < valid) ? a.err2[e0 + j] : 0.0f;
                }
            }
        }


        finish_row<BOUT, SR>(a, e0, valid, acc, e2, red[parity]);
    }
}

// ---------------------------------------------------------------------------
// Eight ranks of 4-bit codes requantised to 4 bits (the W = 8 all-reduce of one
// eight-GPU node) with 16 elements per thread: 256-thread CTAs over the same
// 4096-element rows, each rank's codes of a thread one 8-byte load and one
// scale (blocks of >= 16), and the block statistic, scale, reciprocal and
// loop bookkeeping paid once per 16 elements instead of per 8.  The
// arithmetic per element is that of decode_kernel, so the results are the
// same bits.  Needs 8-byte aligned code pointers and blocks of >= 16 on both
// sides; otherwise decode_kernel runs.
// ---------------------------------------------------------------------------

// REQ = false: the rank sum alone (no requantisation, no stage-2 error): the
// leader's decode of pipeline-A with local quantisation.
// TW > 0: blocks of 16 TW output elements (a team of TW threads), with the
// requantisation as straight-line code (fixed-width butterfly, the clamp chosen
// per warp); TW = 0 reads the team width at run time.
template <int BITS>
__device__ __forceinline__ void rtn8_levels(const float (&v)[8], float s, float y, bool clamp, Packed<BITS>& c,
                                            float (&q)[8])
{
    constexpr float Q = (float)((1 << (BITS - 1)) - 1);
    uint32_t mb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float t = div_by_scale(v[j], s, y);
        if (clamp) t = fminf(fmaxf(t, -Q), Q);
        const float m = __fadd_rn(t, kMagic);                // 1.5*2^23 + rint(t)
        q[j] = __fsub_rn(m, kMagic);
        mb[j] = __float_as_uint(m);
    }
    pack8<BITS>(mb, c);
}

template <bool SR, bool REQ = true, int TW = 0>
__global__ void __launch_bounds__(kThreads16, 3) decode16_w8_kernel(const DecArgs a)
{
    __shared__ float red[2][kThreads16 / 32];
    const int64_t n = a.n;
    const int rows = (int)((n + kRow - 1) / kRow);       // < 2^31 (decode16_fits)
    const int tid = threadIdx.x;
    const Team team = make_team16(REQ ? a.log2Bout : 4);

    uint2 cc[8];
    uint32_t sc[4];                                  // the 8 ranks' fp16 scales, two per word
    auto load = [&](int row) {
        const int64_t e0 = (int64_t)row * kRow + tid * 16;
        if (e0 >= n) return;
        const int64_t off = e0 >> 1;                 // 4-bit codes: 8 bytes per 16 elements
        const int64_t blk = e0 >> a.log2Bin;
#pragma unroll
        for (int k = 0; k < 8; ++k) cc[k] = __ldg(reinterpret_cast<const uint2*>(a.codes[k] + off));
#pragma unroll
        for (int k = 0; k < 4; ++k)
            sc[k] = __byte_perm(__ldg(a.scales[2 * k] + blk), __ldg(a.scales[2 * k + 1] + blk), 0x5410);
    };
    if ((int)blockIdx.x < rows) load(blockIdx.x);
    int parity = 0;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t e0 = (int64_t)row * kRow + tid * 16;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 16 ? 16 : (int)rem);

        float lo[8], hi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) { lo[j] = 0.0f; hi[j] = 0.0f; }
        if (valid > 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                Packed<4> c0, c1;
                c0.w[0] = cc[k].x;
                c1.w[0] = cc[k].y;
                const unsigned short sk = (unsigned short)((k & 1) ? sc[k >> 1] >> 16 : sc[k >> 1] & 0xFFFFu);
                accumulate_rank<4>(c0, sk, k == 0, lo);
                accumulate_rank<4>(c1, sk, k == 0, hi);
            }
        }
        if (row + (int)gridDim.x < rows) load(row + gridDim.x);   // overlaps the requantisation
        if constexpr (!REQ) {
            if (valid == 16) {
                st8_f32(a.sum_out + e0, lo);
                st8_f32(a.sum_out + e0 + 8, hi);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < valid) a.sum_out[e0 + j] = j < 8 ? lo[j] : hi[j - 8];
            }
            continue;
        }
        // the stage-2 error is loaded only now, after the next row's codes are
        // in flight: issued at the top of the row it held 16 registers through
        // the accumulation and measured 8 % slower (0.341 vs 0.317 ms per chunk)
        float e2[16];
        if (a.err2 != nullptr) {
            if (valid == 16) {
                float t0[8], t1[8];
                ld8_f32(a.err2 + e0, t0);
                ld8_f32(a.err2 + e0 + 8, t1);
#pragma unroll
                for (int j = 0; j < 8; ++j) { e2[j] = t0[j]; e2[j + 8] = t1[j]; }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) e2[j] = (j < valid) ? a.err2[e0 + j] : 0.0f;
            }
        }

        if (a.sum_out != nullptr) {
            if (valid == 16) {
                st8_f32(a.sum_out + e0, lo);
                st8_f32(a.sum_out + e0 + 8, hi);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < valid) a.sum_out[e0 + j] = j < 8 ? lo[j] : hi[j - 8];
            }
        }

        // stage-2 error feedback, block statistic over 16 elements, requantise
        float v0[8], v1[8];
        float stat = 0.0f;
        if constexpr (TW > 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v0[j] = lo[j];
                v1[j] = hi[j];
                if (a.err2 != nullptr) { v0[j] = __fadd_rn(v0[j], e2[j]); v1[j] = __fadd_rn(v1[j], e2[j + 8]); }
            }
            if (valid < 16) {                        // the last, partial row only
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j >= valid) v0[j] = 0.0f;
                    if (j + 8 >= valid) v1[j] = 0.0f;
                }
            }
            float mx = max3f(fabsf(v0[0]), fabsf(v0[1]), fabsf(v0[2]));
            mx = max3f(mx, fabsf(v0[3]), fabsf(v0[4]));
            mx = max3f(mx, fabsf(v0[5]), fabsf(v0[6]));
            mx = max3f(mx, fabsf(v0[7]), fabsf(v1[0]));
            mx = max3f(mx, fabsf(v1[1]), fabsf(v1[2]));
            mx = max3f(mx, fabsf(v1[3]), fabsf(v1[4]));
            mx = max3f(mx, fabsf(v1[5]), fabsf(v1[6]));
            stat = fmaxf(mx, fabsf(v1[7]));
            if constexpr (TW <= 16) {
                stat = butterfly<false, TW>(stat);
            } else {
                stat = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(stat)));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float x0 = lo[j], x1 = hi[j];
                if (a.err2 != nullptr) { x0 = __fadd_rn(x0, e2[j]); x1 = __fadd_rn(x1, e2[j + 8]); }
                v0[j] = j < valid ? x0 : 0.0f;
                v1[j] = j + 8 < valid ? x1 : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) stat = fmaxf(stat, fmaxf(fabsf(v0[j]), fabsf(v1[j])));
            stat = team_reduce<false>(stat, team, red[parity]);
        }
        const int64_t blk = e0 >> a.log2Bout;
        const __half sh = block_scale<4>(stat, 1 << a.log2Bout);
        const float s2 = __half2float(sh);
        const float y2 = scale_reciprocal(s2);

        uint32_t rw0[8], rw1[8];
        if constexpr (SR) {
            const uint32_t shift = (uint32_t)(a.index_offset & 3u);
            random_words8(a.index_offset + (uint64_t)e0, a.keys, shift, rw0);
            random_words8(a.index_offset + (uint64_t)e0 + 8, a.keys, shift, rw1);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) { rw0[j] = 0u; rw1[j] = 0u; }
        }
        Packed<4> c0, c1;
        float q0[8], q1[8];
        if constexpr (TW > 0 && !SR) {
            // no clamp where every scale of the warp is normal and below 65504
            // (then |t| < Qmax + 1/2, see quantize8); a zero scale gives t = 0
            if (__all_sync(0xFFFFFFFFu, s2 >= 0x1p-14f && s2 < 65504.0f)) {
                rtn8_levels<4>(v0, s2, y2, false, c0, q0);
                rtn8_levels<4>(v1, s2, y2, false, c1, q1);
            } else {
                rtn8_levels<4>(v0, s2, y2, true, c0, q0);
                rtn8_levels<4>(v1, s2, y2, true, c1, q1);
            }
        } else {
            quantize8<4, SR, false>(v0, s2, y2, rw0, c0, q0);
            quantize8<4, SR, false>(v1, s2, y2, rw1, c1, q1);
        }
        if (e0 < (a.nb_out << a.log2Bout))
            *reinterpret_cast<uint2*>(a.codes_out + (e0 >> 1)) = make_uint2(c0.w[0], c1.w[0]);
        if (team.lane == 0 && blk < a.nb_out) a.scales_out[blk] = __half_as_ushort(sh);

        if (a.err2 != nullptr) {
            float f0[8], f1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                f0[j] = feedback<4>(v0[j], s2, q0[j]);
                f1[j] = feedback<4>(v1[j], s2, q1[j]);
            }
            if (valid == 16) {
                st8_f32(a.err2 + e0, f0);
                st8_f32(a.err2 + e0 + 8, f1);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < valid) a.err2[e0 + j] = j < 8 ? f0[j] : f1[j - 8];
            }
        }
    }
}

// Grids of the decoders (spread_grid in codec.cuh).  Each CTA loads its next
// row while it finishes the current one, so a CTA needs several rows for that
// to pay: on 1.3e9 outputs (sum only) and 1.625e8 (8 -> 4 bits, 8 ranks),
// fractions of measured HBM, one row per CTA measured 0.89-0.90, eight 0.998
// and 1.021-1.026, sixteen 1.005 and 1.002, thirty-two 0.99 and 0.96, against
// 0.983 and 0.994 on a persistent grid.  The requantising 4 -> 4-bit
// 16-element decoder measured the same at eight rows per CTA (0.969) and
// slower at sixteen or more (0.944-0.950), and keeps its persistent grid.
constexpr int kDecSpreadWaves = 12;
constexpr int kDec16SumRowsPerCta = 16;
constexpr int kDec8RowsPerCta = 8;

template <bool SR, bool REQ = true, int TW = 0>
static cudaError_t run_decode16_w8(const DecArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = REQ ? grid_size_threads(decode16_w8_kernel<SR, REQ, TW>, kThreads16, cap, rows)
                         : spread_grid(decode16_w8_kernel<SR, REQ, TW>, kThreads16, cap, rows, kDec16SumRowsPerCta,
                                       kDecSpreadWaves);
    decode16_w8_kernel<SR, REQ, TW><<<grid, kThreads16, 0, st>>>(a);
    return cudaGetLastError();
}

// The rank sum alone through decode16_w8_kernel: eight ranks of 4-bit codes
// in blocks of >= 16, 8-byte aligned code pointers, a sum output.
static bool decode16_sum_fits(const DecArgs& a)
{
    if (a.W != 8 || a.log2Bin < 4 || a.sum_out == nullptr || a.codes_out != nullptr || a.err2 != nullptr ||
        a.n >= ((int64_t)1 << 42))
        return false;
    for (int k = 0; k < 8; ++k)
        if ((reinterpret_cast<uintptr_t>(a.codes[k]) & 7u) != 0) return false;
    return true;
}

static bool decode16_fits(const DecArgs& a)
{
    if (a.W != 8 || a.log2Bin < 4 || a.log2Bout < 4 || a.codes_out == nullptr || a.n >= ((int64_t)1 << 42))
        return false;
    for (int k = 0; k < 8; ++k)
        if ((reinterpret_cast<uintptr_t>(a.codes[k]) & 7u) != 0) return false;
    return (reinterpret_cast<uintptr_t>(a.codes_out) & 7u) == 0;
}

template <int BIN, int BOUT, bool SR, bool MANY, int KW>
static cudaError_t run_decode_kw(const DecArgs& a, cudaStream_t st)
{
    if constexpr (KW == 8 && BIN == 4 && BOUT == 4 && !MANY) {
        if (decode16_fits(a)) {
            switch (a.log2Bout) {
            case 4: return run_decode16_w8<SR, true, 1>(a, st);
            case 5: return run_decode16_w8<SR, true, 2>(a, st);
            case 6: return run_decode16_w8<SR, true, 4>(a, st);
            case 7: return run_decode16_w8<SR, true, 8>(a, st);
            case 8: return run_decode16_w8<SR, true, 16>(a, st);
            case 9: return run_decode16_w8<SR, true, 32>(a, st);
            default: return run_decode16_w8<SR>(a, st);
            }
        }
    }
    if constexpr (KW == 8 && BIN == 4 && BOUT == 0 && !MANY) {
        if (decode16_sum_fits(a)) return run_decode16_w8<false, false>(a, st);
    }
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = spread_grid(decode_kernel<BIN, BOUT, SR, MANY, KW>, kThreads, cap, rows, kDec8RowsPerCta,
                                 kDecSpreadWaves);
    decode_kernel<BIN, BOUT, SR, MANY, KW><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

// DEC_KW selects the instantiations a translation unit compiles: 8 for
// exactly eight ranks, 0 for a rank count read at run time.
template <int BIN, int BOUT, bool SR, bool MANY>
static cudaError_t run_decode(const DecArgs& a, cudaStream_t st)
{
    return run_decode_kw<BIN, BOUT, SR, MANY, (MANY ? 0 : DEC_KW)>(a, st);
}

template <int B, bool MANY>
static cudaError_t decode_same(const DecArgs& a, int bits_out, bool sr, cudaStream_t st)
{
    if (bits_out == 0) return run_decode<B, 0, false, MANY>(a, st);
    if (bits_out != B) return cudaErrorNotSupported;
    if constexpr (B == 1) {
        return run_decode<1, 1, false, MANY>(a, st);
    } else {
        return sr ? run_decode<B, B, true, MANY>(a, st) : run_decode<B, B, false, MANY>(a, st);
    }
}

template <bool MANY>
static cudaError_t decode_dispatch(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    if (bits_in == 8 && bits_out == 4)   // two-level: 8-bit intra stage, 4-bit inter stage
        return sr ? run_decode<8, 4, true, MANY>(a, st) : run_decode<8, 4, false, MANY>(a, st);
    switch (bits_in) {
    case 1: return decode_same<1, MANY>(a, bits_out, sr, st);
    case 2: return decode_same<2, MANY>(a, bits_out, sr, st);
    case 4: return decode_same<4, MANY>(a, bits_out, sr, st);
    case 8: return decode_same<8, MANY>(a, bits_out, sr, st);
    case 12: return decode_same<12, MANY>(a, bits_out, sr, st);
    case 16: return decode_same<16, MANY>(a, bits_out, sr, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace bitscom
