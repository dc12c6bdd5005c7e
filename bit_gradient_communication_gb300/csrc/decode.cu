// decode.cu -- fused decoder kernel for one chunk between the all-to-all and
// the all-gather of a low-bit all-reduce: unpack + dequantise the W ranks'
// codes, sum them in rank order in fp32, optionally add the stage-2 error,
// requantise + repack (bitscom README, "Implemented Features": all-to-all ->
// local reduce -> all-gather; "Backend Registration Options":
// stage2_error_feedback).  Every byte of the W inputs is read once and every
// output byte written once; the rank sum never leaves registers.
#include "codec.cuh"
#include "launch.h"

namespace bitscom {

// BOUT == 0: no requantisation (sum only).
template <int BIN, int BOUT, bool SR>
__global__ void __launch_bounds__(kThreads, (BIN >= 12 || BOUT >= 12) ? 1 : 2) decode_kernel(const DecArgs a)
{
    constexpr int kGroup = 8;   // ranks whose loads are issued together
    __shared__ float red[2][kWarps];
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    const int W = a.W;
    int parity = 0;

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
            for (int w0 = 0; w0 < W; w0 += kGroup) {
                Packed<BIN> c[kGroup];
                float s[kGroup];
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                    if (w0 + k < W) {
                        c[k] = load_codes<BIN>(a.codes[w0 + k], piece);
                        s[k] = __half2float(__ushort_as_half(__ldg(a.scales[w0 + k] + blk_in)));
                    }
                }
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                    if (w0 + k < W) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float d = __fmul_rn(s[k], level_of<BIN>(get_code<BIN>(c[k], j)));
                            acc[j] = (w0 + k == 0) ? d : __fadd_rn(acc[j], d);
                        }
                    }
                }
            }
        }

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
            if (a.err2 != nullptr) {
                if (valid == 8) {
                    float e[8];
                    ld8_f32(a.err2 + e0, e);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = __fadd_rn(acc[j], e[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = (j < valid) ? __fadd_rn(acc[j], a.err2[e0 + j]) : 0.0f;
                }
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
            stat = team_reduce<BOUT == 1>(stat, team, red[parity]);

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
                random_words8(a.index_offset + (uint64_t)e0, a.philox_stream, (uint32_t)a.seed,
                              (uint32_t)(a.seed >> 32), (uint32_t)(a.index_offset & 3u), rw);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) rw[j] = 0u;
            }
            Packed<BOUT> c;
            float q[8];
            quantize8<BOUT, (SR && BOUT > 1)>(v, s2, rw, c, q);

            if (e0 < (a.nb_out << a.log2Bout)) store_codes<BOUT>(a.codes_out, piece, c);
            if (team.lane == 0 && blk < a.nb_out) a.scales_out[blk] = __half_as_ushort(sh);

            if (a.err2 != nullptr) {
                float e[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = __fsub_rn(v[j], __fmul_rn(s2, q[j]));
                if (valid == 8) {
                    st8_f32(a.err2 + e0, e);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) if (j < valid) a.err2[e0 + j] = e[j];
                }
            }
        }
    }
}

template <int BIN, int BOUT, bool SR>
static cudaError_t run_decode(const DecArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = grid_size(decode_kernel<BIN, BOUT, SR>, cap, rows);
    decode_kernel<BIN, BOUT, SR><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int B>
static cudaError_t decode_same(const DecArgs& a, int bits_out, bool sr, cudaStream_t st)
{
    if (bits_out == 0) return run_decode<B, 0, false>(a, st);
    if (bits_out != B) return cudaErrorNotSupported;
    if constexpr (B == 1) {
        return run_decode<1, 1, false>(a, st);
    } else {
        return sr ? run_decode<B, B, true>(a, st) : run_decode<B, B, false>(a, st);
    }
}

cudaError_t launch_decode(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    if (bits_in == 8 && bits_out == 4)   // two-level: 8-bit intra stage, 4-bit inter stage
        return sr ? run_decode<8, 4, true>(a, st) : run_decode<8, 4, false>(a, st);
    switch (bits_in) {
    case 1: return decode_same<1>(a, bits_out, sr, st);
    case 2: return decode_same<2>(a, bits_out, sr, st);
    case 4: return decode_same<4>(a, bits_out, sr, st);
    case 8: return decode_same<8>(a, bits_out, sr, st);
    case 12: return decode_same<12>(a, bits_out, sr, st);
    case 16: return decode_same<16>(a, bits_out, sr, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace bitscom
