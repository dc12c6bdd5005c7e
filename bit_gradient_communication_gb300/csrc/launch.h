// launch.h -- internal interface between the C ABI (api.cpp, sched.cpp) and
// the kernel files.  Not installed; the public interface is include/bitscom.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bitscom.h"

namespace bitscom {

// Philox4x32-10 multipliers and Weyl constants (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11).
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// The key schedule of one launch, expanded on the host so that the kernels
// take every round key from the parameter bank.  Round r uses the key
// (k0 + r W0, k1 + r W1) mod 2^32.  Counter words 2 and 3 are the same for
// every element of a launch (the Philox stream and 0), so the second product
// of the first Philox round is a launch constant too and is folded into the
// two x-terms it feeds: x0 = hi(M1 stream) ^ k0 (first Philox round) and
// x1 = lo(M1 stream) ^ (k0 + W0) (second Philox round).
struct PhiloxKeys {
    uint32_t x0, x1;
    uint32_t k0[10];        // k0 + r W0; Philox rounds r = 2..9 read it
    uint32_t k1[10];        // k1 + r W1
};

inline PhiloxKeys philox_keys(uint64_t seed, uint32_t stream)
{
    PhiloxKeys k;
    const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        k.k0[r] = key0 + (uint32_t)r * kPhiloxW0;
        k.k1[r] = key1 + (uint32_t)r * kPhiloxW1;
    }
    const uint64_t p1 = (uint64_t)kPhiloxM1 * stream;
    k.x0 = (uint32_t)(p1 >> 32) ^ k.k0[0];
    k.x1 = (uint32_t)p1 ^ k.k0[1];
    return k;
}

struct EncArgs {
    const void* x;          // fp32 or bf16 [n]
    float* err;             // [n] or nullptr
    int64_t n;
    int64_t nb;             // ceil(n / B)
    uint8_t* codes;         // packed_bytes(n)
    uint16_t* scales;       // [nb]
    int log2B;
    PhiloxKeys keys;        // stochastic rounding: philox_keys(seed, stream)
    uint64_t index_offset;
    int hadamard;           // 0 or the transform block H
    float* deq = nullptr;   // fused roundtrip only: fl(s*q) as fp32 [n]
    uint32_t pack_mul = 0;  // 2^bits, set by the launcher (packing by multiply-adds)
};

constexpr int kMaxRanks = 64;

struct DecArgs {
    const uint8_t* codes[kMaxRanks];
    const uint16_t* scales[kMaxRanks];
    int W;
    int64_t n;
    int log2Bin;
    int log2Bout;
    int64_t nb_out;
    float* sum_out;         // [n] or nullptr
    float* err2;            // [n] or nullptr
    uint8_t* codes_out;     // or nullptr (no requantisation)
    uint16_t* scales_out;
    PhiloxKeys keys;        // stochastic requantisation: philox_keys(seed, stream)
    uint64_t index_offset;
};

struct DqArgs {
    const uint8_t* codes;
    const uint16_t* scales;
    int64_t n;
    int log2B;
    float mul;
    void* out;              // fp32 or bf16 [n]
    int hadamard;           // 0 or the transform block H (inverse applied)
};

struct SumArgs {
    const void* x[kMaxRanks];   // W arrays of n fp32 or bf16 elements
    int W;
    int64_t n;
    float* out;                 // [n]
};

// Rank-ordered fp32 sum; dtype 0 = fp32, 1 = bf16 inputs.
cudaError_t launch_sum_ranks(const SumArgs& a, int dtype, cudaStream_t st);

// The stochastic encoder without error feedback with 32 elements per thread
// (encode_sr32.cuh): 2- to 16-bit codes, blocks of 32 .. 4096 elements, no
// rotation, codes aligned for one thread's stores (8 bytes at 2 bits, else 16).
inline bool encode32_sr_fits(const EncArgs& a, int bits)
{
    const uintptr_t align = bits == 2 ? 8 : 16;
    return bits >= 2 && a.hadamard == 0 && a.log2B >= 5 && a.log2B <= 12 && a.n < ((int64_t)1 << 42) &&
           (reinterpret_cast<uintptr_t>(a.codes) & (align - 1)) == 0;
}
cudaError_t launch_encode32_sr_f32(const EncArgs& a, int bits, cudaStream_t st);        // 2, 4, 8 bits
cudaError_t launch_encode32_sr_bf16(const EncArgs& a, int bits, cudaStream_t st);
cudaError_t launch_encode32_sr_f32_wide(const EncArgs& a, int bits, cudaStream_t st);   // 12, 16 bits
cudaError_t launch_encode32_sr_bf16_wide(const EncArgs& a, int bits, cudaStream_t st);

// Return cudaErrorNotSupported for a combination without a kernel.
cudaError_t launch_encode_f32(const EncArgs& a, int bits, bool sr, cudaStream_t st);
cudaError_t launch_encode_bf16(const EncArgs& a, int bits, bool sr, cudaStream_t st);
// dtype 0 = fp32, 1 = bf16.
inline cudaError_t launch_encode(const EncArgs& a, int dtype, int bits, bool sr, cudaStream_t st)
{
    return dtype == 0 ? launch_encode_f32(a, bits, sr, st) : launch_encode_bf16(a, bits, sr, st);
}
// bits_out == 0: no requantisation.
cudaError_t launch_decode_few(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st);
cudaError_t launch_decode_w8(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st);
cudaError_t launch_decode_many(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st);
inline cudaError_t launch_decode(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    if (a.W == 8) return launch_decode_w8(a, bits_in, bits_out, sr, st);
    return a.W < 8 ? launch_decode_few(a, bits_in, bits_out, sr, st)
                   : launch_decode_many(a, bits_in, bits_out, sr, st);
}

// Quantise then dequantise in one pass (no error feedback, no rotation):
// codes, scales and a.deq = fl(s*q).  cudaErrorNotSupported when the
// arguments do not fit the one-pass kernel (the caller then runs the encoder
// and the all-gather-side decode).
cudaError_t launch_roundtrip_f32(const EncArgs& a, int bits, bool sr, cudaStream_t st);
cudaError_t launch_roundtrip_bf16(const EncArgs& a, int bits, bool sr, cudaStream_t st);
inline cudaError_t launch_roundtrip(const EncArgs& a, int dtype, int bits, bool sr, cudaStream_t st)
{
    return dtype == 0 ? launch_roundtrip_f32(a, bits, sr, st) : launch_roundtrip_bf16(a, bits, sr, st);
}

// Weight-difference quantisation: a.x = weights, a.err = reference (in/out).
cudaError_t launch_qwd_encode(const EncArgs& a, int dtype, int bits, bool sr, cudaStream_t st);
// wout: 0 none, 1 fp32, 2 bf16.
cudaError_t launch_qwd_apply(const uint8_t* codes, const uint16_t* scales, int64_t n, int log2B,
                             float* ref, void* w_out, int wout, int bits, cudaStream_t st);

// out_dtype 0 = fp32, 1 = bf16.
cudaError_t launch_dequant(const DqArgs& a, int bits, int out_dtype, cudaStream_t st);

// Host-side argument checks of the encoder / decoder entry points (no CUDA
// calls); shared by the plain entry points and the bucket scheduler.
bitscom_status check_encode(const void* x, bitscom_dtype dt, int64_t n, const float* err,
                            const bitscom_qparams* p, const void* codes, const uint16_t* scales);
bitscom_status check_decode(const void* const* codes_in, const uint16_t* const* scales_in, int32_t W,
                            int64_t n, const bitscom_qparams* p_in, const float* sum_out,
                            const float* err2, const bitscom_qparams* p_out, const void* codes_out,
                            const uint16_t* scales_out);
// Remember e as this thread's last CUDA error text (bitscom_last_cuda_error).
const char* record_cuda_error(cudaError_t e);

}  // namespace bitscom
