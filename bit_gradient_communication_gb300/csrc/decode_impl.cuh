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
// scales of ranks 0..7 are loaded while the current row is requantised, and
// the stage-2 error of the current row while its ranks are summed.
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

        // stage-2 error of this row: in flight while the ranks are summed
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

        finish_row<BOUT, SR>(a, e0, valid, acc, e2, red[parity]);
    }
}

template <int BIN, int BOUT, bool SR, bool MANY, int KW>
static cudaError_t run_decode_kw(const DecArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = grid_size(decode_kernel<BIN, BOUT, SR, MANY, KW>, cap, rows);
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
