// Self-check of the codec's quotient v / s (div_by_scale: reciprocal + two
// residual corrections) against CUDA's correctly rounded __fdiv_rn, for every
// positive finite fp16 scale s and n_v values of v per scale: values whose
// quotient lies within 4 ulps of a half-integer or an integer in
// [-32768, 32768] (where rounding decisions are made), random quotients up to
// 2^17, and random finite bit patterns.
// For |v| >= 2^-96 the quotients must be bit-identical; below, the codec only
// uses the quotient's rounding to an integer and its sign.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "codec.cuh"

namespace {

__device__ uint32_t mix32(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)(x ^ (x >> 31));
}

constexpr uint32_t kMaxScale = 0x7BFF;   // largest finite fp16
constexpr int kSlots = 16;

__global__ void probe(uint32_t n_v, unsigned long long* bad, uint32_t* first)
{
    const uint64_t id = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t hi = id / n_v;
    const uint32_t vi = (uint32_t)(id % n_v);
    const uint32_t h = 1u + (uint32_t)hi;
    if (h > kMaxScale) return;
    const float s = __half2float(__ushort_as_half((unsigned short)h));
    const float y = bitscom::scale_reciprocal(s);
    const uint32_t r = mix32(id);
    float v;
    const int kind = vi & 3;
    if (kind == 0) {
        v = __fmul_rn((float)(int32_t)r * 0x1p-14f, s);
    } else if (kind <= 2) {
        const int32_t k = (int32_t)(mix32(id ^ 0x5555u) % 65537u) - 32768;
        const float base = kind == 1 ? (float)k + 0.5f : (float)k;
        v = __fmul_rn(base, s);
        if (v != 0.0f) v = __uint_as_float(__float_as_uint(v) + (uint32_t)((int)((r >> 8) % 9u) - 4));
    } else {
        uint32_t bits = r;
        if (((bits >> 23) & 0xFFu) == 0xFFu) bits &= ~(1u << 30);
        v = __uint_as_float(bits);
    }
    const float ref = __fdiv_rn(v, s);
    const float got = bitscom::div_by_scale(v, s, y);
    bool ok;
    if (!isfinite(ref)) {
        ok = true;   // |v / s| beyond fp32: impossible for a block's own scale
    } else if (fabsf(v) >= 0x1p-96f) {
        ok = __float_as_uint(ref) == __float_as_uint(got);
    } else {
        ok = rintf(ref) == rintf(got) && (ref > 0.0f) == (got > 0.0f) && (ref < 0.0f) == (got < 0.0f);
    }
    if (!ok) {
        const unsigned long long slot = atomicAdd(bad, 1ull);
        if (slot < kSlots) {
            first[3 * slot] = __float_as_uint(v);
            first[3 * slot + 1] = h;
            first[3 * slot + 2] = __float_as_uint(got);
        }
    }
}

}  // namespace

extern "C" int run_division_probe(uint32_t n_v, unsigned long long* bad_out, uint32_t* first_out)
{
    unsigned long long* bad = nullptr;
    uint32_t* first = nullptr;
    if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess) return 1;
    if (cudaMalloc(&first, 3 * kSlots * sizeof(uint32_t)) != cudaSuccess) return 2;
    cudaMemset(bad, 0, sizeof(*bad));
    cudaMemset(first, 0, 3 * kSlots * sizeof(uint32_t));
    const uint64_t total = (uint64_t)kMaxScale * n_v;
    const unsigned threads = 512;
    const uint64_t blocks = (total + threads - 1) / threads;
    probe<<<(unsigned)blocks, threads>>>(n_v, bad, first);
    int rc = cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
    cudaMemcpy(bad_out, bad, sizeof(*bad), cudaMemcpyDeviceToHost);
    cudaMemcpy(first_out, first, 3 * kSlots * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return rc;
}
