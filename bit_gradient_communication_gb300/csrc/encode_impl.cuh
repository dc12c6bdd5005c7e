// encode_impl.cuh -- fused encoder kernel: load g (+ e) -> block statistic ->
// fp16 scale -> quantise -> pack -> store codes, scales and e'.
// One pass over the input: every input byte is read once and every output
// byte written once (bitscom README, "Implemented Features": blockwise
// quantization with per-block FP16 scales; error-feedback in first-stage
// quantization).
#pragma once

#include "codec.cuh"
#include "launch.h"

namespace bitscom {

// One thread's raw inputs for one row: the gradient bits as loaded (fp32, or
// 8 bf16 in a uint4) and the error buffer.  Kept raw so that the loads of the
// next row can be in flight while the current row is computed.
template <int IN, bool EF>
struct RowIn {
    float g[IN == 0 ? 8 : 1];
    uint4 gb;
    float e[EF ? 8 : 1];
};

template <int IN, bool EF>
__device__ __forceinline__ void load_row(const EncArgs& a, int64_t row, RowIn<IN, EF>& r)
{
    const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
    if ((row + 1) * kRow <= a.n) {
        if constexpr (IN == 0) {
            ld8_f32_stream(static_cast<const float*>(a.x) + e0, r.g);
        } else {
            r.gb = ld16_stream(static_cast<const uint16_t*>(a.x) + e0);
        }
        if constexpr (EF) ld8_f32(a.err + e0, r.e);
        return;
    }
    // the last, partial row: element loads, zero fill past n
    const int64_t rem = a.n - e0;
    const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
    uint32_t hb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const bool in = j < valid;
        if constexpr (IN == 0) {
            r.g[j] = in ? static_cast<const float*>(a.x)[e0 + j] : 0.0f;
        } else {
            hb[j] = in ? (uint32_t)static_cast<const uint16_t*>(a.x)[e0 + j] : 0u;
        }
        if constexpr (EF) r.e[j] = in ? a.err[e0 + j] : 0.0f;
    }
    if constexpr (IN == 1) {
        r.gb = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                          hb[6] | (hb[7] << 16));
    }
}

// IN: 0 = fp32, 1 = bf16.  HAD: rotate every a.hadamard-element block of g by
// the Walsh-Hadamard transform before the error is added.  The row loop is
// software-pipelined: the loads of row r + gridDim.x (with error feedback) or
// of row r + 2 gridDim.x (without: two buffers, the loop unrolled by two) are
// issued before row r is computed.
template <int IN, int BITS, bool EF, bool SR, bool HAD>
__global__ void __launch_bounds__(kThreads, 2) encode_kernel(const EncArgs a)
{
    __shared__ float red[2][kWarps];
    const Team team = make_team(a.log2B);
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    const int64_t padded = a.nb << a.log2B;
    const uint32_t shift = (uint32_t)(a.index_offset & 3u);
    const int64_t G = gridDim.x;

    // One row: `cur` holds its inputs and is refilled with row `ahead`.
    auto process = [&](RowIn<IN, EF>& cur, int64_t row, int64_t ahead, int parity) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t piece = e0 >> 3;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        float v[8];
        if constexpr (IN == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = cur.g[j];
        } else {
            bf16x8_to_f32(cur.gb, v);
        }
        if constexpr (HAD) fwht8(v, a.hadamard);
        if constexpr (EF) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 t = __fadd2_rn(make_float2(v[2 * i], v[2 * i + 1]),
                                            make_float2(cur.e[2 * i], cur.e[2 * i + 1]));
                v[2 * i] = t.x;
                v[2 * i + 1] = t.y;
            }
        }
        // prefetch: row `ahead` reuses this buffer; its loads overlap the arithmetic.
        // The memory-bound encoders (error feedback, round to nearest, no
        // rotation) first line up the CTA's warps, so that a row's loads reach
        // DRAM together: 0.956 -> 0.987 of measured HBM for bf16 + EF, 4-bit,
        // block 128.  Issue-bound variants (stochastic rounding, Hadamard,
        // no error feedback) measured slower with the barrier.
        if constexpr (EF && !SR && !HAD) __syncthreads();
        if (ahead < rows) load_row<IN, EF>(a, ahead, cur);

        // block statistic: absmax (b >= 2) or tree sum of |v| (b = 1)
        float stat;
        if constexpr (BITS == 1) {
            stat = __fadd_rn(__fadd_rn(__fadd_rn(fabsf(v[0]), fabsf(v[1])), __fadd_rn(fabsf(v[2]), fabsf(v[3]))),
                             __fadd_rn(__fadd_rn(fabsf(v[4]), fabsf(v[5])), __fadd_rn(fabsf(v[6]), fabsf(v[7]))));
        } else {
            stat = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                         fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
        }
        stat = team_reduce<BITS == 1>(stat, team, red[parity]);

        const int64_t blk = e0 >> a.log2B;
        int n_valid = 1 << a.log2B;
        if constexpr (BITS == 1) {
            const int64_t left = n - (blk << a.log2B);
            if (left < n_valid) n_valid = left > 0 ? (int)left : 1;
        }
        const __half sh = block_scale<BITS>(stat, n_valid);
        const float s = __half2float(sh);

        uint32_t rw[8];
        if constexpr (SR && BITS > 1) {
            random_words8(a.index_offset + (uint64_t)e0, a.keys, shift, rw);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) rw[j] = 0u;
        }
        Packed<BITS> c;
        float q[8];
        quantize8<BITS, (SR && BITS > 1)>(v, s, scale_reciprocal(s), rw, c, q);

        if (e0 < padded) store_codes<BITS>(a.codes, piece, c);
        if (team.lane == 0 && blk < a.nb) a.scales[blk] = __half_as_ushort(sh);

        if constexpr (EF) {
            float e[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = feedback2<BITS>(make_float2(v[2 * i], v[2 * i + 1]), s,
                                                 make_float2(q[2 * i], q[2 * i + 1]));
                e[2 * i] = f.x;
                e[2 * i + 1] = f.y;
            }
            if (valid == 8) {
                st8_f32(a.err + e0, e);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) a.err[e0 + j] = e[j];
            }
        }
    };

    if constexpr (EF) {
        RowIn<IN, EF> cur;
        if ((int64_t)blockIdx.x < rows) load_row<IN, EF>(a, blockIdx.x, cur);
        int parity = 0;
        for (int64_t row = blockIdx.x; row < rows; row += G, parity ^= 1) process(cur, row, row + G, parity);
    } else {
        RowIn<IN, EF> A, B;
        if ((int64_t)blockIdx.x < rows) load_row<IN, EF>(a, blockIdx.x, A);
        if ((int64_t)blockIdx.x + G < rows) load_row<IN, EF>(a, blockIdx.x + G, B);
        for (int64_t row = blockIdx.x; row < rows; row += 2 * G) {
            process(A, row, row + 2 * G, 0);
            if (row + G < rows) process(B, row + G, row + 3 * G, 1);
        }
    }
}

// ---------------------------------------------------------------------------
// 16 elements per thread (1-, 2-, 4-, 8- and 16-bit codes, blocks of >= 16, no
// rotation; used without error feedback, see run_encode): three 256-thread
// CTAs per SM over the same 4096-element rows.  Without the error buffer an
// encoder moves only ~4.3-5 bytes per element, so instruction issue binds
// (stochastic rounding adds two Philox4x32-10 calls per 8 elements); the
// per-row work -- block statistic exchange, scale, reciprocal, index and loop
// bookkeeping -- is paid once per 16 elements.  The per-element arithmetic is that of encode_kernel, so the
// results are the same bits.  Needs code pointers aligned to the 16 codes'
// 2b bytes; otherwise encode_kernel runs.
// ---------------------------------------------------------------------------
template <int IN, bool EF>
struct RowIn16 {
    float g0[IN == 0 ? 8 : 1], g1[IN == 0 ? 8 : 1];
    uint4 gb0, gb1;
    float e0[EF ? 8 : 1], e1[EF ? 8 : 1];
};

template <int IN, bool EF>
__device__ __forceinline__ void load_row16(const EncArgs& a, int row, RowIn16<IN, EF>& r)
{
    const int64_t e0 = (int64_t)row * kRow + threadIdx.x * 16;
    if ((int64_t)(row + 1) * kRow <= a.n) {
        if constexpr (IN == 0) {
            ld8_f32_stream(static_cast<const float*>(a.x) + e0, r.g0);
            ld8_f32_stream(static_cast<const float*>(a.x) + e0 + 8, r.g1);
        } else {
            r.gb0 = ld16_stream(static_cast<const uint16_t*>(a.x) + e0);
            r.gb1 = ld16_stream(static_cast<const uint16_t*>(a.x) + e0 + 8);
        }
        if constexpr (EF) {
            ld8_f32(a.err + e0, r.e0);
            ld8_f32(a.err + e0 + 8, r.e1);
        }
        return;
    }
    // the last, partial row: element loads, zero fill past n
    const int64_t rem = a.n - e0;
    const int valid = rem <= 0 ? 0 : (rem >= 16 ? 16 : (int)rem);
    uint32_t hb[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const bool in = j < valid;
        if constexpr (IN == 0) {
            const float g = in ? static_cast<const float*>(a.x)[e0 + j] : 0.0f;
            if (j < 8) r.g0[j] = g; else r.g1[j - 8] = g;
        } else {
            hb[j] = in ? (uint32_t)static_cast<const uint16_t*>(a.x)[e0 + j] : 0u;
        }
        if constexpr (EF) {
            const float e = in ? a.err[e0 + j] : 0.0f;
            if (j < 8) r.e0[j] = e; else r.e1[j - 8] = e;
        }
    }
    if constexpr (IN == 1) {
        r.gb0 = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                           hb[6] | (hb[7] << 16));
        r.gb1 = make_uint4(hb[8] | (hb[9] << 16), hb[10] | (hb[11] << 16), hb[12] | (hb[13] << 16),
                           hb[14] | (hb[15] << 16));
    }
}

// DEQ: also write fl(s*q) to a.deq (the one-pass roundtrip).
template <int IN, int BITS, bool EF, bool SR, bool DEQ>
__global__ void __launch_bounds__(kThreads16, 3) encode16_kernel(const EncArgs a)
{
    __shared__ float red[2][kThreads16 / 32];
    const Team team = make_team16(a.log2B);
    const int64_t n = a.n;
    const int rows = (int)((n + kRow - 1) / kRow);       // < 2^31 (encode16_fits)
    const uint32_t shift = (uint32_t)(a.index_offset & 3u);
    RowIn16<IN, EF> cur;
    if ((int)blockIdx.x < rows) load_row16<IN, EF>(a, blockIdx.x, cur);
    int parity = 0;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t e0 = (int64_t)row * kRow + threadIdx.x * 16;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 16 ? 16 : (int)rem);
        float v0[8], v1[8];
        if constexpr (IN == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) { v0[j] = cur.g0[j]; v1[j] = cur.g1[j]; }
        } else {
            bf16x8_to_f32(cur.gb0, v0);
            bf16x8_to_f32(cur.gb1, v1);
        }
        if constexpr (EF) {
#pragma unroll
            for (int j = 0; j < 8; ++j) { v0[j] = __fadd_rn(v0[j], cur.e0[j]); v1[j] = __fadd_rn(v1[j], cur.e1[j]); }
        }
        if (row + (int)gridDim.x < rows) load_row16<IN, EF>(a, row + gridDim.x, cur);

        // block statistic: absmax (b >= 2), or for b = 1 the tree sum of |v|
        // over contiguous halves: this thread's 16 elements are two 8-element
        // subtrees, and the butterfly over threads joins contiguous halves
        float stat;
        if constexpr (BITS == 1) {
            auto tree8 = [](const float (&v)[8]) {
                return __fadd_rn(__fadd_rn(__fadd_rn(fabsf(v[0]), fabsf(v[1])), __fadd_rn(fabsf(v[2]), fabsf(v[3]))),
                                 __fadd_rn(__fadd_rn(fabsf(v[4]), fabsf(v[5])), __fadd_rn(fabsf(v[6]), fabsf(v[7]))));
            };
            stat = __fadd_rn(tree8(v0), tree8(v1));
        } else {
            stat = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) stat = fmaxf(stat, fmaxf(fabsf(v0[j]), fabsf(v1[j])));
        }
        // the packed form of stochastic rounding (codes only) tests its pieces
        // for tiny elements here, while the block statistic is exchanged
        constexpr bool kPacked = SR && !EF && !DEQ && (BITS == 2 || BITS == 4);
        bool tiny0 = false, tiny1 = false;
        if constexpr (kPacked) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                tiny0 |= fabsf(v0[j]) < 0x1p-96f;
                tiny1 |= fabsf(v1[j]) < 0x1p-96f;
            }
        }
        stat = team_reduce<BITS == 1>(stat, team, red[parity]);
        const int64_t blk = e0 >> a.log2B;
        int n_valid = 1 << a.log2B;
        if constexpr (BITS == 1) {
            const int64_t left = n - (blk << a.log2B);
            if (left < n_valid) n_valid = left > 0 ? (int)left : 1;
        }
        const __half sh = block_scale<BITS>(stat, n_valid);
        const float s = __half2float(sh);
        const float y = scale_reciprocal(s);

        uint32_t rw0[8], rw1[8];
        if constexpr (SR) {
            random_words16(a.index_offset + (uint64_t)e0, a.keys, shift, rw0, rw1);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) { rw0[j] = 0u; rw1[j] = 0u; }
        }
        Packed<BITS> c0, c1;
        float q0[8], q1[8];
        if constexpr (kPacked) {
            if (s >= 0x1p-14f && s < 65504.0f) {      // a normal, unsaturated scale
                quantize8_sr_packed<BITS>(v0, s, y, rw0, tiny0, a.pack_mul, c0);
                quantize8_sr_packed<BITS>(v1, s, y, rw1, tiny1, a.pack_mul, c1);
            } else {
                quantize8<BITS, SR>(v0, s, y, rw0, c0, q0);
                quantize8<BITS, SR>(v1, s, y, rw1, c1, q1);
            }
        } else {
            quantize8<BITS, SR>(v0, s, y, rw0, c0, q0);
            quantize8<BITS, SR>(v1, s, y, rw1, c1, q1);
        }
        if (e0 < (a.nb << a.log2B)) {
            uint8_t* p = a.codes + e0 * BITS / 8;
            if constexpr (BITS == 1) {
                *reinterpret_cast<uint16_t*>(p) = (uint16_t)((c0.w[0] & 0xFFu) | ((c1.w[0] & 0xFFu) << 8));
            } else if constexpr (BITS == 2) {
                *reinterpret_cast<uint32_t*>(p) = (c0.w[0] & 0xFFFFu) | (c1.w[0] << 16);
            } else if constexpr (BITS == 4) {
                *reinterpret_cast<uint2*>(p) = make_uint2(c0.w[0], c1.w[0]);
            } else if constexpr (BITS == 8) {
                *reinterpret_cast<uint4*>(p) = make_uint4(c0.w[0], c0.w[1], c1.w[0], c1.w[1]);
            } else {
                uint4* q = reinterpret_cast<uint4*>(p);
                q[0] = make_uint4(c0.w[0], c0.w[1], c0.w[2], c0.w[3]);
                q[1] = make_uint4(c1.w[0], c1.w[1], c1.w[2], c1.w[3]);
            }
        }
        if (team.lane == 0 && blk < a.nb) a.scales[blk] = __half_as_ushort(sh);

        if constexpr (DEQ) {
            // fl(s*q): exact for b <= 12, one rounding at b = 16, as in the decoders
            float d0[8], d1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) { d0[j] = __fmul_rn(s, q0[j]); d1[j] = __fmul_rn(s, q1[j]); }
            if (valid == 16) {
                st8_f32(a.deq + e0, d0);
                st8_f32(a.deq + e0 + 8, d1);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < valid) a.deq[e0 + j] = j < 8 ? d0[j] : d1[j - 8];
            }
        }

        if constexpr (EF) {
            float f0[8], f1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                f0[j] = feedback<BITS>(v0[j], s, q0[j]);
                f1[j] = feedback<BITS>(v1[j], s, q1[j]);
            }
            if (valid == 16) {
                st8_f32(a.err + e0, f0);
                st8_f32(a.err + e0 + 8, f1);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < valid) a.err[e0 + j] = j < 8 ? f0[j] : f1[j - 8];
            }
        }
    }
}

// Grids of the encoders (spread_grid): about this many rows per CTA when the
// launch spans at least kEncSpreadWaves waves of resident CTAs, else the
// persistent grid.  Measured on 1.3e9 bf16 and 2^28 fp32 elements (L2
// flushed, fractions of measured HBM), against the persistent grid:
//   16-element kernel, error feedback, round to nearest: 2 rows per CTA,
//     every width and block 1.05 (0.97-0.99 persistent with the 8-element
//     kernel, 0.90-0.95 persistent with this one); 3 rows 1.04, 8 rows 1.03;
//   16-element kernel without error feedback: 8 rows per CTA, fp32 4-bit
//     0.95 (0.88), 16-bit 1.01 (1.00), bf16 4-bit 0.89 (0.82);
//   8-element kernel with error feedback (stochastic rounding, the rotated
//     encoders, 12-bit codes): 8 rows per CTA, fp32 2- and 4-bit stochastic
//     rounding 1.03 (0.93), bf16 2-bit 0.997 (0.96), 8-bit with Hadamard
//     H = 128 0.992 (0.972); 3-4 rows per CTA measured up to 1.04 on the fp32
//     cases but 0.96-0.97 on the bf16 and rotated ones.  Without error
//     feedback (its two-buffer loop, read-heavy: fp32 12-bit codes) it stays
//     persistent: 8 rows per CTA measured 0.91-1.00 against 0.93-1.02.
// On 5e7 elements the 16-element error-feedback kernel at 2 rows per CTA
// (13 waves) still won (0.960 against 0.937); 8 rows per CTA of the 8-element
// kernel (5 waves) lost (0.893).
constexpr int kEncSpreadWaves = 12;
constexpr int kEnc16EfRowsPerCta = 2;
constexpr int kEnc16RowsPerCta = 8;
constexpr int kEnc8RowsPerCta = 8;

// The memory-bound round-to-nearest encoders of 4- to 16-bit codes without
// error feedback measured faster on a persistent grid with three CTAs per SM
// than with the four their registers allow (fp32, 2^28 elements: 16-bit 1.01
// against 0.86-0.91 of measured HBM, 4- and 8-bit 0.97-0.98 against
// 0.95-0.96); 1- and 2-bit codes run as many as fit.
template <bool SR, bool DEQ, int BITS>
constexpr int enc16_occ_cap() { return (!SR && !DEQ && BITS >= 4) ? 3 : 0; }

// The 16-element kernel takes round to nearest with error feedback only over
// a spread grid: on a persistent grid it measured below the 8-element kernel
// (5e7 elements 0.872 against 0.937; fp32 25 MiB buckets 0.59-0.64 against
// 0.65-0.70).
template <int IN, int BITS>
static bool encode16_ef_spreads(const EncArgs& a)
{
    static std::atomic<int> res{0};
    const int c = resident_ctas(encode16_kernel<IN, BITS, true, false, false>, kThreads16, res,
                                enc16_occ_cap<false, false, BITS>());
    const int64_t rows = (a.n + kRow - 1) / kRow;
    return (rows + kEnc16EfRowsPerCta - 1) / kEnc16EfRowsPerCta >= (int64_t)kEncSpreadWaves * c;
}

template <int IN, int BITS, bool EF, bool SR, bool DEQ = false>
static cudaError_t run_encode16(const EncArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = spread_grid(encode16_kernel<IN, BITS, EF, SR, DEQ>, kThreads16, cap, rows,
                                 EF ? kEnc16EfRowsPerCta : kEnc16RowsPerCta, kEncSpreadWaves,
                                 enc16_occ_cap<SR, DEQ, BITS>());
    EncArgs b = a;
    b.pack_mul = BITS <= 8 ? (1u << BITS) : 0u;
    encode16_kernel<IN, BITS, EF, SR, DEQ><<<grid, kThreads16, 0, st>>>(b);
    return cudaGetLastError();
}

inline bool encode16_fits(const EncArgs& a, int bits)
{
    return a.hadamard == 0 && a.log2B >= 4 && a.n < ((int64_t)1 << 42) &&
           (reinterpret_cast<uintptr_t>(a.codes) & (uintptr_t)(2 * bits - 1)) == 0;
}

template <int IN, int BITS, bool EF, bool SR, bool HAD>
static cudaError_t run_encode_h(const EncArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};   // SMs x resident CTAs of this instantiation
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = EF ? spread_grid(encode_kernel<IN, BITS, EF, SR, HAD>, kThreads, cap, rows, kEnc8RowsPerCta,
                                      kEncSpreadWaves)
                        : grid_size(encode_kernel<IN, BITS, EF, SR, HAD>, cap, rows);
    encode_kernel<IN, BITS, EF, SR, HAD><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

// The Hadamard rotation has instantiations for 2-, 4- and 8-bit codes.
template <int IN, int BITS, bool EF, bool SR>
static cudaError_t run_encode(const EncArgs& a, cudaStream_t st)
{
    if constexpr (SR && !EF && BITS >= 2) {
        if (encode32_sr_fits(a, BITS)) {
            if constexpr (BITS >= 12)
                return IN == 0 ? launch_encode32_sr_f32_wide(a, BITS, st) : launch_encode32_sr_bf16_wide(a, BITS, st);
            else
                return IN == 0 ? launch_encode32_sr_f32(a, BITS, st) : launch_encode32_sr_bf16(a, BITS, st);
        }
    }
    if constexpr (!EF && BITS != 12) {
        if (encode16_fits(a, BITS)) return run_encode16<IN, BITS, EF, SR>(a, st);
    }
    // error feedback with round to nearest: the 16-element kernel when the
    // launch is large enough for a spread grid (with stochastic rounding it
    // spills: 1.01 against 1.04 for the 8-element kernel on 2^28 fp32)
    if constexpr (EF && !SR && BITS != 12) {
        if (encode16_fits(a, BITS) && encode16_ef_spreads<IN, BITS>(a))
            return run_encode16<IN, BITS, true, false>(a, st);
    }
    if (a.hadamard == 0) return run_encode_h<IN, BITS, EF, SR, false>(a, st);
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
        return run_encode_h<IN, BITS, EF, SR, true>(a, st);
    } else {
        return cudaErrorNotSupported;
    }
}

template <int IN, int BITS>
static cudaError_t encode_bits(const EncArgs& a, bool sr, cudaStream_t st)
{
    const bool ef = a.err != nullptr;
    if constexpr (BITS == 1) {
        return ef ? run_encode<IN, 1, true, false>(a, st) : run_encode<IN, 1, false, false>(a, st);
    } else {
        if (ef) return sr ? run_encode<IN, BITS, true, true>(a, st) : run_encode<IN, BITS, true, false>(a, st);
        return sr ? run_encode<IN, BITS, false, true>(a, st) : run_encode<IN, BITS, false, false>(a, st);
    }
}

template <int IN, int BITS>
static cudaError_t roundtrip_bits(const EncArgs& a, bool sr, cudaStream_t st)
{
    if (!encode16_fits(a, BITS)) return cudaErrorNotSupported;
    if constexpr (BITS == 1) {
        return run_encode16<IN, 1, false, false, true>(a, st);
    } else {
        return sr ? run_encode16<IN, BITS, false, true, true>(a, st) : run_encode16<IN, BITS, false, false, true>(a, st);
    }
}

template <int IN>
static cudaError_t roundtrip_dispatch(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    if (a.err != nullptr || a.deq == nullptr) return cudaErrorNotSupported;
    switch (bits) {
    case 1: return roundtrip_bits<IN, 1>(a, sr, st);
    case 2: return roundtrip_bits<IN, 2>(a, sr, st);
    case 4: return roundtrip_bits<IN, 4>(a, sr, st);
    case 8: return roundtrip_bits<IN, 8>(a, sr, st);
    case 16: return roundtrip_bits<IN, 16>(a, sr, st);
    default: return cudaErrorNotSupported;
    }
}

template <int IN>
static cudaError_t encode_dispatch(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    switch (bits) {
    case 1: return encode_bits<IN, 1>(a, sr, st);
    case 2: return encode_bits<IN, 2>(a, sr, st);
    case 4: return encode_bits<IN, 4>(a, sr, st);
    case 8: return encode_bits<IN, 8>(a, sr, st);
    case 12: return encode_bits<IN, 12>(a, sr, st);
    case 16: return encode_bits<IN, 16>(a, sr, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace bitscom
