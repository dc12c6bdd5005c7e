// launch.h -- internal interface between the C ABI (api.cpp, sched.cpp) and
// the kernel files.  Not installed; the public interface is include/bitscom.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bitscom.h"

namespace bitscom {

struct EncArgs {
    const void* x;          // fp32 or bf16 [n]
    float* err;             // [n] or nullptr
    int64_t n;
    int64_t nb;             // ceil(n / B)
    uint8_t* codes;         // packed_bytes(n)
    uint16_t* scales;       // [nb]
    int log2B;
    uint32_t philox_stream;
    uint64_t seed;
    uint64_t index_offset;
    int hadamard;           // 0 or the transform block H
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
    uint32_t philox_stream;
    uint64_t seed;
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
