// dequant.cu -- all-gather-side decode: after the all-gather of a low-bit
// all-reduce every rank holds the requantised chunks of all ranks (bitscom
// README, "Implemented Features": all-to-all -> local reduce -> all-gather)
// and turns them back into its gradient: out = fl(fl(s*q) * mul), written as
// fp32 or bf16 (round to nearest even).  One read of the codes and scales,
// one write of the output.
//
// Three kernels.  dequant16_kernel (blocks of >= 16, no rotation, codes and
// output aligned for its wider accesses) decodes 16 elements per thread with
// 32-byte stores over a grid of many short-lived CTAs; dequant32h_kernel
// takes the rotated decode when the blocks hold >= 32 elements (32 elements
// per thread, so up to five of the transform's stages stay in registers);
// dequant_kernel takes every other case, 8 elements per thread over a
// persistent grid with the row loop software-pipelined like the encoder's.
#include <cuda_bf16.h>

#include "codec.cuh"
#include "launch.h"
#include "wide16.cuh"

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

// ---------------------------------------------------------------------------
// 16 elements per thread (wide16.cuh).  The decode writes 4-16x the bytes it
// reads; each CTA decodes about three rows (the next row's codes loaded before
// the current row's store) and the grid holds rows / 3 CTAs, never fewer than
// the GPU holds at once: every width into bf16 or fp32, 2^29 and 1.3e9
// elements, 0.98-1.04 of measured HBM (the persistent 8-element kernel
// 0.60-0.98; one or two rows per CTA 0.77-0.94 for 1-bit codes, 8 rows
// 0.96-1.03; a ring of rows in registers and 512-thread CTAs made no
// difference).
constexpr int kDq16RowsPerCta = 3;

// y = fl(fl(s*q) * mul) for one piece.  s*q is exact in fp32 for every width
// (an fp16 scale times a level of at most 16 bits), so the packed-fp16 levels
// with the mixed-precision fma and the fp32 levels with a multiply give the
// same bits as the single rounding of the oracle.
template <int BITS>
__device__ __forceinline__ void piece_values(const Packed<BITS>& c, unsigned short s, float mul, float (&y)[8])
{
    float d[8];
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
        uint32_t h[4];
        level_pairs<BITS>(c, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            d[pair_lo<BITS>(i)] = fma_f16(s, (unsigned short)(h[i] & 0xFFFFu), -0.0f);
            d[pair_hi<BITS>(i)] = fma_f16(s, (unsigned short)(h[i] >> 16), -0.0f);
        }
    } else {
        const float sf = __half2float(__ushort_as_half(s));
        float l[8];
        levels8<BITS>(c, l);
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(sf, l[j]);
    }
    const float2 mul2 = make_float2(mul, mul);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __fmul2_rn(make_float2(d[2 * i], d[2 * i + 1]), mul2);
        y[2 * i] = t.x;
        y[2 * i + 1] = t.y;
    }
}

// Thread t of a CTA decodes elements [16t, 16t + 16) of rows blockIdx.x + k G.
template <int BITS, int OUT>
__global__ void __launch_bounds__(kWideThreads) dequant16_kernel(const DqArgs a)
{
    const int64_t n = a.n;
    const int64_t rows = (n + kWideRow - 1) / kWideRow;
    const int64_t G = gridDim.x;
    Codes16<BITS> c{};
    unsigned short s = 0;
    auto load = [&](int64_t row) {
        const int64_t e0 = row * kWideRow + (int64_t)threadIdx.x * 16;
        if (row >= rows || e0 >= n) return;
        c = load_codes16<BITS>(a.codes, e0);
        s = __ldg(a.scales + (e0 >> a.log2B));
    };
    load(blockIdx.x);
    for (int64_t row = blockIdx.x; row < rows; row += G) {
        const int64_t e0 = row * kWideRow + (int64_t)threadIdx.x * 16;
        float y0[8], y1[8];
        piece_values<BITS>(c.c[0], s, a.mul, y0);
        piece_values<BITS>(c.c[1], s, a.mul, y1);
        load(row + G);
        if (e0 >= n) continue;
        const int64_t rem = n - e0;
        if constexpr (OUT == 0) {
            float* out = static_cast<float*>(a.out) + e0;
            if (rem >= 16) {
                st8_f32(out, y0);
                st8_f32(out + 8, y1);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) if (j < rem) out[j] = j < 8 ? y0[j] : y1[j - 8];
            }
        } else {
            uint16_t* out = static_cast<uint16_t*>(a.out) + e0;
            if (rem >= 16) {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[i] = bf16_pair(y0[2 * i], y0[2 * i + 1]);
                    w[4 + i] = bf16_pair(y1[2 * i], y1[2 * i + 1]);
                }
                st8_b32(out, w);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < rem) out[j] = __bfloat16_as_ushort(__float2bfloat16_rn(j < 8 ? y0[j] : y1[j - 8]));
            }
        }
    }
}

template <int BITS>
static bool dq16_fits(const DqArgs& a)
{
    return a.hadamard == 0 && a.log2B >= 4 &&
           (reinterpret_cast<uintptr_t>(a.codes) & (code16_align<BITS>() - 1)) == 0 &&
           (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
}

template <int BITS, int OUT>
static cudaError_t run_dequant16(const DqArgs& a, cudaStream_t st)
{
    static std::atomic<int> resident{0};
    const int64_t rows = (a.n + kWideRow - 1) / kWideRow;
    const int grid = spread_grid(dequant16_kernel<BITS, OUT>, kWideThreads, resident, rows, kDq16RowsPerCta, 1);
    dequant16_kernel<BITS, OUT><<<grid, kWideThreads, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The rotated decode with 32 elements per thread (blocks of >= 32).  The inverse
// transform is the forward one (stages h = 1, 2, ..., H/2, pair (i, i + h)
// -> (x_i + x_{i+h}, x_i - x_{i+h})) followed by the exact factor 1/H, as in
// fwht8.  With 8 elements per thread every stage from h = 8 on is a round of
// xor shuffles, one per element, and each round measured ~62 us per 2^29
// elements: H = 128 into bf16 took 478 us, 0.42 of measured HBM.  Here the
// stages h = 1..16 (up to H/2 for H = 8 and 16) run in registers on packed
// pairs and only log2(H/32) rounds cross threads, each a shuffle per element and one packed fma per
// pair (k x + o with k = +1 on the lower lane and -1 on the upper: the same
// single rounding as x + o and o - x).  bf16 output is stored directly, one
// 32-byte store per 16 elements; fp32 output goes through shared memory so
// that every store instruction of a warp writes 1 KB contiguous (the direct
// 128 bytes per thread measured 0.72-0.84 of measured HBM, the staged stores
// 0.97-0.99).  2^29 elements, bf16 / fp32 out: H = 32 0.97 / 0.98, 64 0.87 /
// 0.98, 128 0.75-0.88 / 0.98-0.99, 256 0.56 / 0.82 (the 8-element kernel
// 0.57 / 0.88, 0.48 / 0.77, 0.42-0.51 / 0.69-0.78, 0.32 / 0.61).  Staging the
// bf16 stores measured slower (0.67-0.95): there the shuffles and the
// arithmetic, not the stores, set the pace.
constexpr int kH32Threads = 256;
constexpr int kH32Row = kH32Threads * 32;
constexpr int kH32RowsPerCta = 4;
constexpr int kH32StageWords = 36;                  // padded row of the fp32 staging buffer

template <int BITS>
struct Codes32h { Packed<BITS> c[4]; };

// codes of 32 consecutive elements (e0 a multiple of 32): 8, 16 or 32 bytes
template <int BITS>
__device__ __forceinline__ Codes32h<BITS> load_codes32(const uint8_t* codes, int64_t e0)
{
    Codes32h<BITS> t;
    const uint8_t* p = codes + (e0 >> 3) * BITS;
    if constexpr (BITS == 2) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        t.c[0].w[0] = w.x & 0xFFFFu; t.c[1].w[0] = w.x >> 16;
        t.c[2].w[0] = w.y & 0xFFFFu; t.c[3].w[0] = w.y >> 16;
    } else if constexpr (BITS == 4) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        t.c[0].w[0] = w.x; t.c[1].w[0] = w.y; t.c[2].w[0] = w.z; t.c[3].w[0] = w.w;
    } else {
        const uint4* q = reinterpret_cast<const uint4*>(p);
        const uint4 w0 = __ldg(q), w1 = __ldg(q + 1);
        t.c[0].w[0] = w0.x; t.c[0].w[1] = w0.y; t.c[1].w[0] = w0.z; t.c[1].w[1] = w0.w;
        t.c[2].w[0] = w1.x; t.c[2].w[1] = w1.y; t.c[3].w[0] = w1.z; t.c[3].w[1] = w1.w;
    }
    return t;
}

// one in-register stage of span HS over 32 values, two butterflies per pair
// of packed instructions (a + b, and a - b as the fma -b + a)
template <int HS>
__device__ __forceinline__ void wht_stage32(float (&x)[32])
{
    const float2 m1 = make_float2(-1.0f, -1.0f);
    if constexpr (HS == 1) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float2 a = make_float2(x[j], x[j + 2]), b = make_float2(x[j + 1], x[j + 3]);
            const float2 s = __fadd2_rn(a, b), d = __ffma2_rn(b, m1, a);
            x[j] = s.x; x[j + 2] = s.y; x[j + 1] = d.x; x[j + 3] = d.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            if (j & HS) continue;
            const float2 a = make_float2(x[j], x[j + 1]), b = make_float2(x[j + HS], x[j + HS + 1]);
            const float2 s = __fadd2_rn(a, b), d = __ffma2_rn(b, m1, a);
            x[j] = s.x; x[j + 1] = s.y; x[j + HS] = d.x; x[j + HS + 1] = d.y;
        }
    }
}

// Thread t decodes elements [32t, 32t + 32) of rows blockIdx.x + k G.  n is a
// multiple of H.  SMALL = false (H >= 32): the H/32 threads of a transform
// block are all in or all out of range, and out-of-range threads still take
// part in the shuffles.  SMALL = true (H = 8 or 16): no stage crosses threads,
// and the last thread may hold whole transform blocks beyond n, which it
// computes from the padding of its codes block and does not store.  (One
// kernel for both, with the stages and the ragged stores chosen at run time,
// took 68-74 registers and measured 0.61 instead of 0.75 for H = 128.)
template <int BITS, int OUT, bool SMALL>
__global__ void __launch_bounds__(kH32Threads) dequant32h_kernel(const DqArgs a)
{
    __shared__ __align__(16) float stage[OUT == 0 ? kH32Threads * kH32StageWords : 4];
    const int64_t n = a.n;
    const int64_t rows = (n + kH32Row - 1) / kH32Row;
    const int lane = threadIdx.x & 31;
    const int H = a.hadamard;
    const float inv = 1.0f / (float)H;                         // a power of two: exact
    const float2 inv2 = make_float2(inv, inv), mul2 = make_float2(a.mul, a.mul);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t e0 = row * kH32Row + (int64_t)threadIdx.x * 32;
        const bool active = e0 < n;
        float v[32];
        if (active) {
            const Codes32h<BITS> c = load_codes32<BITS>(a.codes, e0);
            const unsigned short s = __ldg(a.scales + (e0 >> a.log2B));     // blocks of >= H >= 32
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t h[4];
                level_pairs<BITS>(c.c[p], h);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[8 * p + pair_lo<BITS>(i)] = fma_f16(s, (unsigned short)(h[i] & 0xFFFFu), -0.0f);
                    v[8 * p + pair_hi<BITS>(i)] = fma_f16(s, (unsigned short)(h[i] >> 16), -0.0f);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
        }
        wht_stage32<1>(v);
        wht_stage32<2>(v);
        wht_stage32<4>(v);
        if constexpr (SMALL) {
            if (H == 16) wht_stage32<8>(v);
        } else {
            wht_stage32<8>(v);
            wht_stage32<16>(v);
        }
        for (int m = 1; m < (SMALL ? 1 : (H >> 5)); m <<= 1) {
            const float k = (lane & m) ? -1.0f : 1.0f;
            const float2 k2 = make_float2(k, k);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float o0 = __shfl_xor_sync(0xFFFFFFFFu, v[j], m);
                const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v[j + 1], m);
                const float2 r = __ffma2_rn(make_float2(v[j], v[j + 1]), k2, make_float2(o0, o1));
                v[j] = r.x;
                v[j + 1] = r.y;
            }
        }
        // out = fl(fl(d / H) * mul), each rounded as the scalar multiply
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float2 t = __fmul2_rn(__fmul2_rn(make_float2(v[j], v[j + 1]), inv2), mul2);
            v[j] = t.x;
            v[j + 1] = t.y;
        }
        if constexpr (OUT == 0) {
            // lane l's 32 values into row l of its warp's buffer, then store
            // instruction q takes elements [256 q, 256 q + 256) of the warp's
            // 1024 (row 8q + l/4, words 8 (l % 4) .. + 8); the padded rows keep
            // both the writes and the reads free of bank conflicts
            float* buf = stage + (threadIdx.x >> 5) * (32 * kH32StageWords);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(buf + lane * kH32StageWords + 4 * i) =
                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            __syncwarp();
            const int64_t wbase = row * kH32Row + (int64_t)(threadIdx.x & ~31) * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float* src = buf + (8 * q + (lane >> 2)) * kH32StageWords + 8 * (lane & 3);
                const float4 t0 = *reinterpret_cast<const float4*>(src);
                const float4 t1 = *reinterpret_cast<const float4*>(src + 4);
                const float w[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                const int64_t o = wbase + 256 * q + 8 * lane;
                if (!SMALL || o + 8 <= n) {
                    if (o < n) st8_f32(static_cast<float*>(a.out) + o, w);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) if (o + j < n) static_cast<float*>(a.out)[o + j] = w[j];
                }
            }
            __syncwarp();
        } else {
            if (!active) continue;
            uint16_t* out = static_cast<uint16_t*>(a.out) + e0;
            if (!SMALL || e0 + 32 <= n) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = bf16_pair(v[16 * q + 2 * i], v[16 * q + 2 * i + 1]);
                    st8_b32(out + 16 * q, w);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (e0 + j < n) out[j] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
            }
        }
    }
}

template <int BITS>
static bool dq32h_fits(const DqArgs& a)
{
    constexpr uintptr_t ca = BITS == 2 ? 8 : 16;
    return a.hadamard >= 8 && a.log2B >= 5 && (reinterpret_cast<uintptr_t>(a.codes) & (ca - 1)) == 0 &&
           (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
}

template <int BITS, int OUT, bool SMALL>
static cudaError_t run_dequant32h_s(const DqArgs& a, cudaStream_t st)
{
    static std::atomic<int> resident{0};
    const int64_t rows = (a.n + kH32Row - 1) / kH32Row;
    const int grid =
        spread_grid(dequant32h_kernel<BITS, OUT, SMALL>, kH32Threads, resident, rows, kH32RowsPerCta, 1);
    dequant32h_kernel<BITS, OUT, SMALL><<<grid, kH32Threads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int BITS, int OUT>
static cudaError_t run_dequant32h(const DqArgs& a, cudaStream_t st)
{
    return a.hadamard >= 32 ? run_dequant32h_s<BITS, OUT, false>(a, st) : run_dequant32h_s<BITS, OUT, true>(a, st);
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
    if (dq16_fits<BITS>(a)) return run_dequant16<BITS, OUT>(a, st);
    if (a.hadamard == 0) return run_dequant_h<BITS, OUT, false>(a, st);
    if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
        if (dq32h_fits<BITS>(a)) return run_dequant32h<BITS, OUT>(a, st);
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
