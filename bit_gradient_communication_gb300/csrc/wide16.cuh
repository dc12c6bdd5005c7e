// wide16.cuh -- pieces shared by the streaming kernels that decode 16
// elements per thread in 256-thread CTAs over a grid of short-lived CTAs
// (spread_grid in codec.cuh): the all-gather-side decode and the
// weight-difference apply.  The 16-element code load, the 32-byte store and
// the bf16 pair packing.
#pragma once

#include <cuda_bf16.h>

#include "codec.cuh"

namespace bitscom {

constexpr int kWideThreads = 256;
constexpr int kWideRow = kWideThreads * 16;     // elements per CTA row

// Codes of 16 consecutive elements (two 8-element pieces), one load of 2b
// bytes (two for 12 and 16 bits).  e0 is a multiple of 16 below n: with
// blocks of >= 16 the packed codes cover whole blocks, so all 16 elements'
// codes are inside the buffer even when n ends inside them.
template <int BITS>
struct Codes16 { Packed<BITS> c[2]; };

template <int BITS>
__device__ __forceinline__ Codes16<BITS> load_codes16(const uint8_t* codes, int64_t e0)
{
    Codes16<BITS> t;
    const uint8_t* p = codes + (e0 >> 3) * BITS;
    if constexpr (BITS == 1) {
        const uint32_t w = __ldg(reinterpret_cast<const unsigned short*>(p));
        t.c[0].w[0] = w & 0xFFu;
        t.c[1].w[0] = w >> 8;
    } else if constexpr (BITS == 2) {
        const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
        t.c[0].w[0] = w & 0xFFFFu;
        t.c[1].w[0] = w >> 16;
    } else if constexpr (BITS == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        t.c[0].w[0] = w.x;
        t.c[1].w[0] = w.y;
    } else if constexpr (BITS == 8) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        t.c[0].w[0] = w.x; t.c[0].w[1] = w.y;
        t.c[1].w[0] = w.z; t.c[1].w[1] = w.w;
    } else if constexpr (BITS == 12) {
        const uint2* q = reinterpret_cast<const uint2*>(p);
        const uint2 w0 = __ldg(q), w1 = __ldg(q + 1), w2 = __ldg(q + 2);
        t.c[0].w[0] = w0.x; t.c[0].w[1] = w0.y; t.c[0].w[2] = w1.x;
        t.c[1].w[0] = w1.y; t.c[1].w[1] = w2.x; t.c[1].w[2] = w2.y;
    } else {
        const uint4* q = reinterpret_cast<const uint4*>(p);
        const uint4 w0 = __ldg(q), w1 = __ldg(q + 1);
        t.c[0].w[0] = w0.x; t.c[0].w[1] = w0.y; t.c[0].w[2] = w0.z; t.c[0].w[3] = w0.w;
        t.c[1].w[0] = w1.x; t.c[1].w[1] = w1.y; t.c[1].w[2] = w1.z; t.c[1].w[3] = w1.w;
    }
    return t;
}

// Code alignment the 16-element loads need: twice the 8-element piece's
// load width (two 8-byte loads for 12 bits).
template <int BITS>
__host__ __device__ constexpr uintptr_t code16_align()
{
    return BITS == 1 ? 2 : (BITS == 2 ? 4 : (BITS == 4 ? 8 : (BITS == 12 ? 8 : 16)));
}

// one 32-byte store of eight words (p 32-byte aligned)
__device__ __forceinline__ void st8_b32(void* p, const uint32_t (&w)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
                    "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// two fp32 values as a bf16 pair (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi)
{
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

}  // namespace bitscom
