// dequant.cu -- all-gather-side decode: after the all-gather of a low-bit
// all-reduce every rank holds the requantised chunks of all ranks (bitscom
// README, "Implemented Features": all-to-all -> local reduce -> all-gather)
// and turns them back into its gradient: out = fl(fl(s*q) * mul), written as
// fp32 or bf16 (round to nearest even).  One read of the codes and scales,
// one write of the output; the row loop is software-pipelined like the
// encoder's.
#include <cuda_bf16.h>

#include "codec.cuh"
#include "launch.h"

namespace bitscom {

// Rows of codes in flight per thread.  The codes are only b/8 bytes per
// element, so with one row ahead a decode of <= 8-bit codes into bf16 keeps
// only ~6-12 KB of reads in flight per SM; a ring of four rows in registers
// took it from 0.75-0.87 to 0.85-0.95 of measured HBM (2-, 4-, 8-bit codes,
// 2^29 elements; 1-bit codes take the same ring).  fp32 output (twice the
// writes, and the per-row barrier below) measured best with one row ahead, as
// did 16- and 12-bit codes (12-bit into bf16, 2^29 elements: 0.87-0.88 of
// measured HBM with one row, 0.78-0.79 with the four-row ring).
template <int BITS, int OUT>
__host__ __device__ constexpr int dq_depth() { return (OUT == 1 && BITS <= 8) ? 4 : 1; }

// OUT: 0 = fp32, 1 = bf16.  HAD: inverse Walsh-Hadamard rotation of every
// a.hadamard-element block (the same transform, then the exact factor 1/H).
// Thread t of a CTA decodes elements [8t, 8t + 8) of rows blockIdx.x + k G
// (G = gridDim.x); row r + D G is loaded into ring slot r's registers as soon
// as row r's levels are formed.
template <int BITS, int OUT, bool HAD>
__global__ void __launch_bounds__(kThreads, 2) dequant_kernel(const DqArgs a)
{
    constexpr int D = dq_depth<BITS, OUT>();
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    const int64_t G = gridDim.x;
    Packed<BITS> ring[D];
    unsigned short ring_s[D];
    auto load = [&](int k, int64_t row) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        if ((D > 1 && row >= rows) || e0 >= n) return;
        ring[k] = load_codes<BITS>(a.codes, e0 >> 3);
        ring_s[k] = __ldg(a.scales + (e0 >> a.log2B));
    };
    // decode row `row` from ring slot k, refilling the slot with row + D G
    auto process = [&](int k, int64_t row) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        float d[8];
        if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
            uint32_t h[4];
            level_pairs<BITS>(ring[k], h);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                d[pair_lo<BITS>(i)] = fma_f16(ring_s[k], (unsigned short)(h[i] & 0xFFFFu), -0.0f);
                d[pair_hi<BITS>(i)] = fma_f16(ring_s[k], (unsigned short)(h[i] >> 16), -0.0f);
            }
        } else {
            const float s = __half2float(__ushort_as_half(ring_s[k]));
            float l[8];
            levels8<BITS>(ring[k], l);
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(s, l[j]);
        }
        // fp32 output from codes of >= 4 bits: line up the CTA's warps so that
        // the row's loads and stores reach DRAM together (4-bit, block 128:
        // 0.85 -> 0.87; 16-bit 0.85 -> 0.92); for bf16 output and 1-2-bit codes
        // the barrier measured slower
        if constexpr (OUT == 0 && BITS >= 4) __syncthreads();
        if constexpr (D == 1) {
            if (row + G < rows) load(0, row + G);
        } else {
            load(k, row + D * G);                    // checks the row itself
        }
        if constexpr (HAD) {
            fwht8(d, a.hadamard);
            const float inv = 1.0f / (float)a.hadamard;          // a power of two: exact
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(d[j], inv);
        }
        // out = fl(d * mul); the bf16 decodes of narrow codes (the ring
        // kernels, partly issue-bound) take two lanes per instruction (each
        // rounded as __fmul_rn: 2-bit 0.85 -> 0.87 of measured HBM), the others
        // measured best with the scalar multiply
        float y[8];
        if constexpr (D > 1) {
            const float2 mul2 = make_float2(a.mul, a.mul);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 t = __fmul2_rn(make_float2(d[2 * i], d[2 * i + 1]), mul2);
                y[2 * i] = t.x;
                y[2 * i + 1] = t.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(d[j], a.mul);
        }
        if constexpr (OUT == 0) {
            float* out = static_cast<float*>(a.out);
            if (valid == 8) {
                st8_f32(out + e0, y);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) out[e0 + j] = y[j];
            }
        } else {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
            if (valid == 8) {
                uint4 w;
                __nv_bfloat162 p0 = __floats2bfloat162_rn(y[0], y[1]), p1 = __floats2bfloat162_rn(y[2], y[3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(y[4], y[5]), p3 = __floats2bfloat162_rn(y[6], y[7]);
                w.x = *reinterpret_cast<uint32_t*>(&p0);
                w.y = *reinterpret_cast<uint32_t*>(&p1);
                w.z = *reinterpret_cast<uint32_t*>(&p2);
                w.w = *reinterpret_cast<uint32_t*>(&p3);
                *reinterpret_cast<uint4*>(out + e0) = w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) out[e0 + j] = __float2bfloat16_rn(y[j]);
            }
        }
    };
    if constexpr (D == 1) {
        if ((int64_t)blockIdx.x < rows) load(0, blockIdx.x);
        for (int64_t row = blockIdx.x; row < rows; row += G) process(0, row);
    } else {
#pragma unroll
        for (int k = 0; k < D; ++k) {
            ring[k] = Packed<BITS>{};
            ring_s[k] = 0;
            load(k, (int64_t)blockIdx.x + k * G);
        }
        for (int64_t base = blockIdx.x; base < rows; base += D * G) {
#pragma unroll
            for (int k = 0; k < D; ++k) {
                const int64_t row = base + k * G;
                if (row >= rows) break;                  // uniform over the CTA
                process(k, row);
            }
        }
    }
}

template <int BITS, int OUT, bool HAD>
static cudaError_t run_dequant_h(const DqArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = grid_size(dequant_kernel<BITS, OUT, HAD>, cap, rows);
    dequant_kernel<BITS, OUT, HAD><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int BITS, int OUT>
static cudaError_t run_dequant(const DqArgs& a, cudaStream_t st)
{
    if (a.hadamard == 0) return run_dequant_h<BITS, OUT, false>(a, st);
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
        return run_dequant_h<BITS, OUT, true>(a, st);
    } else {
        return cudaErrorNotSupported;
    }
}

template <int OUT>
static cudaError_t dequant_bits(const DqArgs& a, int bits, cudaStream_t st)
{
    switch (bits) {
    case 1: return run_dequant<1, OUT>(a, st);
    case 2: return run_dequant<2, OUT>(a, st);
    case 4: return run_dequant<4, OUT>(a, st);
    case 8: return run_dequant<8, OUT>(a, st);
    case 12: return run_dequant<12, OUT>(a, st);
    case 16: return run_dequant<16, OUT>(a, st);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_dequant(const DqArgs& a, int bits, int out_dtype, cudaStream_t st)
{
    return out_dtype == 0 ? dequant_bits<0>(a, bits, st) : dequant_bits<1>(a, bits, st);
}

}  // namespace bitscom
