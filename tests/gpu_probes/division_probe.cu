// Self-check of the codec's quotient v / s (div_by_scale: reciprocal + one
// residual correction) against CUDA's correctly rounded __fdiv_rn, for every
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

// RN(1/s) of every positive finite fp16 value against __frcp_rn.
__global__ void recip_probe(unsigned long long* bad, uint32_t* first)
{
    const uint32_t h = 1u + blockIdx.x * blockDim.x + threadIdx.x;
    if (h > kMaxScale) return;
    const float s = __half2float(__ushort_as_half((unsigned short)h));
    const float got = bitscom::scale_reciprocal(s), ref = __frcp_rn(s);
    if (__float_as_uint(got) != __float_as_uint(ref)) {
        const unsigned long long slot = atomicAdd(bad, 1ull);
        if (slot < kSlots) { first[3 * slot] = h; first[3 * slot + 1] = __float_as_uint(got); first[3 * slot + 2] = __float_as_uint(ref); }
    }
}

// The fp16 block scale from every fp32 absmax bit pattern in [lo, hi) against
// fp16_rne(min(__fdiv_rn(absmax, Qmax), 65504)), and the fp32 quotient itself
// against __fdiv_rn.
template <int BITS>
__global__ void scale_probe(uint32_t lo, uint32_t hi, unsigned long long* bad, uint32_t* first)
{
    constexpr float Q = (float)((1 << (BITS - 1)) - 1);
    constexpr float yQ = (float)(1.0 / (double)((1 << (BITS - 1)) - 1));
    for (uint64_t u = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < hi;
         u += (uint64_t)gridDim.x * blockDim.x) {
        const float stat = __uint_as_float((uint32_t)u);
        const __half got = bitscom::block_scale<BITS>(stat, 8);
        const __half ref = __float2half_rn(fminf(__fdiv_rn(stat, Q), 65504.0f));
        const bool q_ok = __float_as_uint(bitscom::div_by_scale(stat, Q, yQ)) == __float_as_uint(__fdiv_rn(stat, Q));
        if (__half_as_ushort(got) != __half_as_ushort(ref) || !q_ok) {
            const unsigned long long slot = atomicAdd(bad, 1ull);
            if (slot < kSlots) { first[3 * slot] = (uint32_t)u; first[3 * slot + 1] = BITS; first[3 * slot + 2] = __half_as_ushort(got); }
        }
    }
}

}  // namespace

// which: 0 = reciprocal of every fp16 scale, 1 = block scale over [2^-100, 2^100).
extern "C" int run_scale_probe(int which, unsigned long long* bad_out, uint32_t* first_out)
{
    unsigned long long* bad = nullptr;
    uint32_t* first = nullptr;
    if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess) return 1;
    if (cudaMalloc(&first, 3 * kSlots * sizeof(uint32_t)) != cudaSuccess) return 2;
    cudaMemset(bad, 0, sizeof(*bad));
    cudaMemset(first, 0, 3 * kSlots * sizeof(uint32_t));
    if (which == 0) {
        recip_probe<<<(kMaxScale + 255) / 256, 256>>>(bad, first);
    } else {
        const uint32_t lo = 0x0D800000u, hi = 0x71800000u;   // [2^-100, 2^100)
        scale_probe<2><<<4096, 512>>>(lo, hi, bad, first);
        scale_probe<4><<<4096, 512>>>(lo, hi, bad, first);
        scale_probe<8><<<4096, 512>>>(lo, hi, bad, first);
        scale_probe<12><<<4096, 512>>>(lo, hi, bad, first);
        scale_probe<16><<<4096, 512>>>(lo, hi, bad, first);
    }
    int rc = cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
    cudaMemcpy(bad_out, bad, sizeof(*bad), cudaMemcpyDeviceToHost);
    cudaMemcpy(first_out, first, 3 * kSlots * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return rc;
}

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
