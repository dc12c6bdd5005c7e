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

// OUT: 0 = fp32, 1 = bf16.  HAD: inverse Walsh-Hadamard rotation of every
// a.hadamard-element block (the same transform, then the exact factor 1/H).
template <int BITS, int OUT, bool HAD>
__global__ void __launch_bounds__(kThreads, 2) dequant_kernel(const DqArgs a)
{
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    Packed<BITS> cur;
    unsigned short cur_s = 0;
    auto load = [&](int64_t row) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        if (e0 >= n) return;
        cur = load_codes<BITS>(a.codes, e0 >> 3);
        cur_s = __ldg(a.scales + (e0 >> a.log2B));
    };
    if ((int64_t)blockIdx.x < rows) load(blockIdx.x);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        float d[8];
        if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
            uint32_t h[4];
            level_pairs<BITS>(cur, h);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                d[pair_lo<BITS>(i)] = fma_f16(cur_s, (unsigned short)(h[i] & 0xFFFFu), -0.0f);
                d[pair_hi<BITS>(i)] = fma_f16(cur_s, (unsigned short)(h[i] >> 16), -0.0f);
            }
        } else {
            const float s = __half2float(__ushort_as_half(cur_s));
            float l[8];
            levels8<BITS>(cur, l);
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(s, l[j]);
        }
        // fp32 output from codes of >= 4 bits: line up the CTA's warps so that
        // the row's loads and stores reach DRAM together (4-bit, block 128:
        // 0.85 -> 0.87; 16-bit 0.85 -> 0.92); for bf16 output and 1-2-bit codes
        // the barrier measured slower
        if constexpr (OUT == 0 && BITS >= 4) __syncthreads();
        if (row + gridDim.x < rows) load(row + gridDim.x);   // prefetch the next row
        if constexpr (HAD) {
            fwht8(d, a.hadamard);
            const float inv = 1.0f / (float)a.hadamard;          // a power of two: exact
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(d[j], inv);
        }
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(d[j], a.mul);
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
