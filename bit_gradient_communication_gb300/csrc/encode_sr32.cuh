// encode_sr32.cuh -- the stochastic-rounding encoder without error feedback,
// 32 elements per thread, for 2- to 16-bit codes and blocks of 32 to 4096
// elements (bitscom README, "Implemented Features": blockwise quantization
// with per-block FP16 scales, stochastic rounding support).
//
// The codes are those of encode16_kernel; the layout is organised around the
// cost of the arithmetic rather than of the memory traffic.  Philox4x32-10
// (one counter per four elements) keeps the FMA-heavy pipe busy, the block
// statistic and the packing the ALU pipe; the ways they are combined here:
//   * each row of a thread is one basic block: the Philox runs, the absmax
//     and minimum, the team butterfly (its width a template parameter), the
//     scale, the packed quantisation and the stores are straight-line code,
//     so that the compiler interleaves the multiply-bound and the ALU-bound
//     instructions within every warp.  Two quantisers cover every scale:
//     the one-sided clamp with the packed-word fix (quantize8_sr_packed)
//     where every scale of the warp is at least one_sided_min_scale and
//     below 65504, else the two-sided clamp (quantize8_sr_clamped), chosen
//     per warp (12- and 16-bit codes always take the two-sided one).  Teams
//     of a warp or more reduce with redux.sync; wider teams add a per-team
//     named barrier, and run their first Philox counters before it.  The
//     cases neither quantiser covers -- an element with 0 < |v| < 2^-96,
//     an index offset not a multiple of 4, a Philox counter whose low word
//     wraps inside the thread's run -- are tested together at the end of the
//     row, which is then recomputed on the general path (random_words8,
//     quantize8);
//   * 32 elements per thread (8192-element rows of a 256-thread CTA) spread
//     the per-row work (team butterfly, scale and reciprocal, the rare-case
//     test, addresses, the scale store) over twice the elements of
//     encode16_kernel and store each thread's codes in one or two 16-byte
//     stores;
//   * the loop is unrolled by two with alternating input registers, so that
//     the prefetched row needs no register copies.
// Measured on 2^28 fp32 Laplace values, 4-bit codes, block 128: 246.4 us
// (0.724 of measured HBM) against 293.5 us for encode16_kernel.
#pragma once

#include <type_traits>

#include "codec.cuh"
#include "launch.h"

namespace bitscom {

constexpr int kThreads32 = 256;
constexpr int kRow32 = kThreads32 * 32;      // elements per CTA row

// One thread's raw inputs for one row: 32 fp32 values, or 32 bf16 values
// (four 16-byte words).
template <int IN>
struct RowIn32 {
    float g[IN == 0 ? 32 : 1];
    uint4 gb[IN == 0 ? 1 : 4];
};

// A full row's inputs: vector loads.
template <int IN>
__device__ __forceinline__ void load_full32(const EncArgs& a, uint64_t e0, RowIn32<IN>& r)
{
    if constexpr (IN == 0) {
        const float* x = static_cast<const float*>(a.x) + e0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float t[8];
            ld8_f32_stream(x + 8 * q, t);
#pragma unroll
            for (int j = 0; j < 8; ++j) r.g[8 * q + j] = t[j];
        }
    } else {
        const uint16_t* x = static_cast<const uint16_t*>(a.x) + e0;
#pragma unroll
        for (int q = 0; q < 4; ++q) r.gb[q] = ld16_stream(x + 8 * q);
    }
}

// The last, partial row: element loads, zero fill past n.
template <int IN>
__device__ __forceinline__ void load_part32(const EncArgs& a, uint64_t e0, RowIn32<IN>& r)
{
    const int64_t rem = a.n - (int64_t)e0;
    const int valid = rem <= 0 ? 0 : (rem >= 32 ? 32 : (int)rem);
    if constexpr (IN == 0) {
        const float* x = static_cast<const float*>(a.x) + e0;
#pragma unroll
        for (int j = 0; j < 32; ++j) r.g[j] = j < valid ? x[j] : 0.0f;
    } else {
        const uint16_t* x = static_cast<const uint16_t*>(a.x) + e0;
        uint32_t h[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = j < valid ? x[j] : 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            r.gb[q] = make_uint4(h[8 * q] | (h[8 * q + 1] << 16), h[8 * q + 2] | (h[8 * q + 3] << 16),
                                 h[8 * q + 4] | (h[8 * q + 5] << 16), h[8 * q + 6] | (h[8 * q + 7] << 16));
    }
}

// The smallest fp16 scale s for which quantize8_sr_packed's one-sided clamp
// holds: 2^(b-1) 2^-24.  For a normal s the fp16 rounding of x = RN(absmax /
// Qmax) is within 2^-11 relative; for a subnormal s it is within 2^-25, and
// with x >= s - 2^-25 >= (2 Qmax + 1) 2^-25 the block's |t| stays below
// (Qmax + 1/2)(1 + 2^-24) < Qmax + 1.  So t > -Qmax - 1, stochastic rounding
// falls at most to -Qmax - 1, and the packed-word fix (offset code 0 -> 1)
// gives the clamp.  Smaller, zero or saturated (65504) scales take the
// two-sided clamp (quantize8_sr_clamped).
template <int BITS>
__device__ __forceinline__ constexpr float one_sided_min_scale()
{
    return (float)(1 << (BITS - 1)) * 0x1p-24f;
}

// Place piece p's packed codes (8 elements) into the thread's code words
// (codes of up to 8 bits; wider ones are stored as they are packed).
template <int BITS>
__device__ __forceinline__ void put_piece(uint32_t (&cw)[BITS], int p, const Packed<BITS>& c)
{
    static_assert(BITS <= 8, "codes of up to 8 bits");
    if constexpr (BITS == 2) {
        if (p & 1) cw[p >> 1] |= c.w[0] << 16;
        else cw[p >> 1] = c.w[0] & 0xFFFFu;
    } else {
        constexpr int K = BITS / 4;            // words per piece: 1 or 2
#pragma unroll
        for (int k = 0; k < K; ++k) cw[K * p + k] = c.w[k];
    }
}

// Store two pieces' codes (16 elements) of 12 or 16 bits: 24 bytes at an
// 8-byte boundary, or 32 at a 16-byte one.
template <int BITS>
__device__ __forceinline__ void store_two_pieces(uint8_t* p, const Packed<BITS>& c0, const Packed<BITS>& c1)
{
    if constexpr (BITS == 12) {
        uint2* o = reinterpret_cast<uint2*>(p);
        o[0] = make_uint2(c0.w[0], c0.w[1]);
        o[1] = make_uint2(c0.w[2], c1.w[0]);
        o[2] = make_uint2(c1.w[1], c1.w[2]);
    } else {
        uint4* o = reinterpret_cast<uint4*>(p);
        o[0] = make_uint4(c0.w[0], c0.w[1], c0.w[2], c0.w[3]);
        o[1] = make_uint4(c1.w[0], c1.w[1], c1.w[2], c1.w[3]);
    }
}

// One thread's row: elements e0 .. e0+31, a team of TW threads per block;
// PART: the last, partial row (stores only within the blocks).
template <int IN, int BITS, int TW, bool PART>
__device__ __forceinline__ void sr32_row(const EncArgs& a, const RowIn32<IN>& r, uint64_t e0, float* red)
{
    float v[32];
    if constexpr (IN == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = r.g[j];
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float t[8];
            bf16x8_to_f32(r.gb[q], t);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[8 * q + j] = t[j];
        }
    }
    const uint64_t i0 = a.index_offset + e0;
    const uint64_t g = i0 >> 2;

    // block absmax (and this thread's smallest magnitude, for the rare test)
    float mx = max3f(fabsf(v[0]), fabsf(v[1]), fabsf(v[2]));
    float mn = min3f(fabsf(v[0]), fabsf(v[1]), fabsf(v[2]));
#pragma unroll
    for (int j = 3; j < 31; j += 2) {
        mx = max3f(mx, fabsf(v[j]), fabsf(v[j + 1]));
        mn = min3f(mn, fabsf(v[j]), fabsf(v[j + 1]));
    }
    float stat = fmaxf(mx, fabsf(v[31]));
    mn = fminf(mn, fabsf(v[31]));
    // teams wider than a warp wait at a barrier below: the first Philox run
    // goes before it, where it can overlap the exchange
    constexpr bool kEarly = TW > 32;
    uint4 w_early[kEarly ? 4 : 1];
    if constexpr (kEarly) philox10_run<4>((uint32_t)g, (uint32_t)(g >> 32), a.keys, w_early);
    if constexpr (TW <= 16) {
        stat = butterfly<false, TW>(stat);
    } else {
        // the maximum of non-negative floats is that of their bit patterns
        stat = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(stat)));
        if constexpr (TW > 32) {
            // teams of TW/32 warps: per-warp maxima through shared memory
            // (red: this row's slots), one named barrier per team (ids 1..)
            constexpr int kWarpsPerTeam = TW / 32;
            const int team = threadIdx.x / TW;
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = stat;
            asm volatile("bar.sync %0, %1;" :: "r"(1 + team), "n"(TW) : "memory");
            stat = red[team * kWarpsPerTeam];
#pragma unroll
            for (int k = 1; k < kWarpsPerTeam; ++k) stat = fmaxf(stat, red[team * kWarpsPerTeam + k]);
        }
    }
    const __half sh = block_scale<BITS>(stat, 1 << a.log2B);
    const float s = __half2float(sh);
    const float y = scale_reciprocal(s);

    // Philox words and packed codes, elements 16h .. 16h+15: the one-sided
    // clamp (quantize8_sr_packed) when every scale of the warp allows it,
    // else the two-sided one (quantize8_sr_clamped); the choice is uniform
    // over the warp, so the branch does not diverge.  Codes of up to 8 bits
    // are collected and stored at the end of the row; 12- and 16-bit codes
    // (the two-sided clamp always) are stored per 16 elements, which keeps
    // fewer registers live, and stored again if the row is redone.
    // (the destination is formed where it is used: kept live across the
    // quantisation it cost the narrow codes ~1.5 %)
    auto write = [&]() { return !PART || (int64_t)e0 < (a.nb << a.log2B); };
    auto out = [&]() { return a.codes + (e0 >> 3) * BITS; };
    uint32_t cw[BITS <= 8 ? BITS : 1];
    auto quantize_row = [&](auto two_sided) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 w[4];
            const uint64_t gh = g + 4 * h;
            if (kEarly && h == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) w[k] = w_early[kEarly ? k : 0];
            } else {
                philox10_run<4>((uint32_t)gh, (uint32_t)(gh >> 32), a.keys, w);
            }
            const uint32_t rw0[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
            const uint32_t rw1[8] = {w[2].x, w[2].y, w[2].z, w[2].w, w[3].x, w[3].y, w[3].z, w[3].w};
            float v0[8], v1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v0[j] = v[16 * h + j];
                v1[j] = v[16 * h + 8 + j];
            }
            Packed<BITS> c0, c1;
            if constexpr (decltype(two_sided)::value || BITS >= 12) {
                quantize8_sr_clamped<BITS>(v0, s, y, rw0, a.pack_mul, c0);
                quantize8_sr_clamped<BITS>(v1, s, y, rw1, a.pack_mul, c1);
            } else {
                quantize8_sr_packed<BITS>(v0, s, y, rw0, false, a.pack_mul, c0);
                quantize8_sr_packed<BITS>(v1, s, y, rw1, false, a.pack_mul, c1);
            }
            if constexpr (BITS <= 8) {
                put_piece<BITS>(cw, 2 * h, c0);
                put_piece<BITS>(cw, 2 * h + 1, c1);
            } else if (write()) {
                store_two_pieces<BITS>(out() + 2 * h * BITS, c0, c1);
            }
        }
    };
    if constexpr (BITS >= 12) {
        quantize_row(std::true_type{});
    } else if (__all_sync(0xFFFFFFFFu, s >= one_sided_min_scale<BITS>() && s < 65504.0f)) {
        quantize_row(std::false_type{});
    } else {
        quantize_row(std::true_type{});
    }
    // the smallest magnitude also flags zeros, which the fast quotient divides
    // exactly: rows flagged only by zeros keep their codes
    const bool words_off = (((uint32_t)i0 & 3u) != 0) | ((uint32_t)g > 0xFFFFFFF8u);
    bool redo = words_off;
    if (mn < 0x1p-96f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) redo |= fabsf(v[j]) < 0x1p-96f && v[j] != 0.0f;
    }
    if (redo) {
        const uint32_t shift = (uint32_t)i0 & 3u;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t rw[8];
            random_words8(i0 + 8 * p, a.keys, shift, rw);
            float vp[8], q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) vp[j] = v[8 * p + j];
            Packed<BITS> c;
            quantize8<BITS, true>(vp, s, y, rw, c, q);
            if constexpr (BITS <= 8) {
                put_piece<BITS>(cw, p, c);
            } else if (write()) {
                uint32_t* o = reinterpret_cast<uint32_t*>(out() + p * BITS);
#pragma unroll
                for (int k = 0; k < BITS / 4; ++k) o[k] = c.w[k];
            }
        }
    }
    if constexpr (BITS <= 8) {
        if (write()) {
            uint8_t* const o = out();
            if constexpr (BITS == 2) {
                *reinterpret_cast<uint2*>(o) = make_uint2(cw[0], cw[1]);
            } else {
#pragma unroll
                for (int k = 0; k < BITS / 4; ++k)
                    reinterpret_cast<uint4*>(o)[k] = make_uint4(cw[4 * k], cw[4 * k + 1], cw[4 * k + 2], cw[4 * k + 3]);
            }
        }
    }
    const int64_t blk = (int64_t)(e0 >> a.log2B);
    if ((threadIdx.x & (TW - 1)) == 0 && (!PART || blk < a.nb)) a.scales[blk] = __half_as_ushort(sh);
}

template <int IN, int BITS, int TW>
__global__ void __launch_bounds__(kThreads32, 2) encode32_sr_kernel(const EncArgs a)
{
    // row counts fit in 32 bits (n < 2^42); the element offsets take 64
    const int full = (int)(a.n / kRow32);                 // full rows
    const int G = gridDim.x;
    const uint64_t step = (uint64_t)G * kRow32;
    int row = blockIdx.x;
    uint64_t e0 = (uint64_t)row * kRow32 + threadIdx.x * 32;
    // per-warp maxima of teams wider than a warp: one set of slots per
    // alternate row, a third for the partial row (a warp may reach the next
    // row's exchange only after every warp of its team has read this one's)
    __shared__ float red[3][kThreads32 / 32];
    RowIn32<IN> ra, rb;
    if (row < full) load_full32<IN>(a, e0, ra);
    while (row < full) {
        if (row + G < full) load_full32<IN>(a, e0 + step, rb);
        sr32_row<IN, BITS, TW, false>(a, ra, e0, red[0]);
        row += G;
        e0 += step;
        if (row >= full) break;
        if (row + G < full) load_full32<IN>(a, e0 + step, ra);
        sr32_row<IN, BITS, TW, false>(a, rb, e0, red[1]);
        row += G;
        e0 += step;
    }
    // the partial last row, by the CTA whose turn it is
    if (a.n % kRow32 != 0 && full % G == (int)blockIdx.x) {
        const uint64_t ep = (uint64_t)full * kRow32 + threadIdx.x * 32;
        load_part32<IN>(a, ep, ra);
        sr32_row<IN, BITS, TW, true>(a, ra, ep, red[2]);
    }
}

template <int IN, int BITS, int TW>
static cudaError_t run_encode32_tw(const EncArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};   // SMs x resident CTAs
    const int64_t rows = (a.n + kRow32 - 1) / kRow32;
    int c = cap.load(std::memory_order_relaxed);
    if (c == 0) {
        int dev = 0, occ = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode32_sr_kernel<IN, BITS, TW>, kThreads32, 0);
        c = (sms > 0 ? sms : 1) * (occ > 0 ? occ : 1);
        cap.store(c, std::memory_order_relaxed);
    }
    const int grid = (int)(rows < c ? rows : c);
    EncArgs b = a;
    b.pack_mul = 1u << BITS;
    encode32_sr_kernel<IN, BITS, TW><<<grid, kThreads32, 0, st>>>(b);
    return cudaGetLastError();
}

// Launch for blocks of 32 .. 4096 elements (encode32_sr_fits, launch.h).
template <int IN, int BITS>
static cudaError_t run_encode32_sr(const EncArgs& a, cudaStream_t st)
{
    switch (a.log2B) {
    case 5: return run_encode32_tw<IN, BITS, 1>(a, st);
    case 6: return run_encode32_tw<IN, BITS, 2>(a, st);
    case 7: return run_encode32_tw<IN, BITS, 4>(a, st);
    case 8: return run_encode32_tw<IN, BITS, 8>(a, st);
    case 9: return run_encode32_tw<IN, BITS, 16>(a, st);
    case 10: return run_encode32_tw<IN, BITS, 32>(a, st);
    case 11: return run_encode32_tw<IN, BITS, 64>(a, st);
    case 12: return run_encode32_tw<IN, BITS, 128>(a, st);
    default: return cudaErrorNotSupported;
    }
}

// 2-, 4- and 8-bit codes, and 12- and 16-bit codes: instantiated in separate
// translation units (compile time).
template <int IN>
static cudaError_t encode32_sr_bits_narrow(const EncArgs& a, int bits, cudaStream_t st)
{
    switch (bits) {
    case 2: return run_encode32_sr<IN, 2>(a, st);
    case 4: return run_encode32_sr<IN, 4>(a, st);
    case 8: return run_encode32_sr<IN, 8>(a, st);
    default: return cudaErrorNotSupported;
    }
}

template <int IN>
static cudaError_t encode32_sr_bits_wide(const EncArgs& a, int bits, cudaStream_t st)
{
    switch (bits) {
    case 12: return run_encode32_sr<IN, 12>(a, st);
    case 16: return run_encode32_sr<IN, 16>(a, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace bitscom
