// qwd.cu -- weight-difference quantisation for the sharded weight all-gather
// (SDP4Bit README, "Weight Quantization Arguments": --quantized-weights,
// --weight-quantization-bits, --wq-group-size; overview: "quantization on
// weight differences").
//   sender   d = fl(w - ref) is quantised (codes, fp16 scales) and the shard
//            owner's reference advances: ref = fl(ref + fl(s*q));
//   receiver every rank applies the gathered codes to its own reference copy
//            the same way (optionally writing the weights as fp32 or bf16), so
//            all copies stay bit-identical and the residual w - ref carries
//            over to the next step.
// The encoder and the 8-element apply use the row / piece / team
// decomposition of codec.cuh and are software-pipelined like the encoder; the
// 16-element apply (blocks of >= 16, codes and weights aligned for its wider
// accesses) runs over a grid of short-lived CTAs (wide16.cuh).
#include <cuda_bf16.h>

#include "encode_impl.cuh"
#include "wide16.cuh"

namespace bitscom {

// fl(ref + fl(s*q)) in one rounding: s*q (fp16 scale x level, at most 22
// significant bits for b <= 8) is exact in fp32.
__device__ __forceinline__ float advance(float ref, float s, float q) { return __fmaf_rn(s, q, ref); }

template <int IN, int BITS, bool SR>
__global__ void __launch_bounds__(kThreads, 2) qwd_encode_kernel(const EncArgs a)
{
    __shared__ float red[2][kWarps];
    const Team team = make_team(a.log2B);
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    const int64_t padded = a.nb << a.log2B;
    const uint32_t shift = (uint32_t)(a.index_offset & 3u);
    float* ref = a.err;
    int parity = 0;

    RowIn<IN, true> cur;   // g and the reference (in the error slot)
    if ((int64_t)blockIdx.x < rows) load_row<IN, true>(a, blockIdx.x, cur);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t piece = e0 >> 3;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        float v[8], r[8];
        if constexpr (IN == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = cur.g[j];
        } else {
            bf16x8_to_f32(cur.gb, v);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            r[j] = cur.e[j];
            v[j] = __fsub_rn(v[j], r[j]);   // the weight difference
        }
        __syncthreads();   // the CTA's next-row loads reach DRAM together (0.970 -> 0.981)
        if (row + gridDim.x < rows) load_row<IN, true>(a, row + gridDim.x, cur);

        float stat = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                           fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
        stat = team_reduce<false>(stat, team, red[parity]);
        const int64_t blk = e0 >> a.log2B;
        const __half sh = block_scale<BITS>(stat, 1 << a.log2B);
        const float s = __half2float(sh);
        uint32_t rw[8];
        if constexpr (SR) {
            random_words8(a.index_offset + (uint64_t)e0, a.keys, shift, rw);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) rw[j] = 0u;
        }
        Packed<BITS> c;
        float q[8];
        quantize8<BITS, SR>(v, s, scale_reciprocal(s), rw, c, q);
        if (e0 < padded) store_codes<BITS>(a.codes, piece, c);
        if (team.lane == 0 && blk < a.nb) a.scales[blk] = __half_as_ushort(sh);

        float out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) out[j] = advance(r[j], s, q[j]);
        if (valid == 8) {
            st8_f32(ref + e0, out);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) if (j < valid) ref[e0 + j] = out[j];
        }
    }
}

struct QwdApplyArgs {
    const uint8_t* codes;
    const uint16_t* scales;
    int64_t n;
    int log2B;
    float* ref;
    void* w_out;            // fp32 or bf16 [n], or nullptr
};

// WOUT: 0 = no weight copy, 1 = fp32, 2 = bf16.
template <int BITS, int WOUT>
__global__ void __launch_bounds__(kThreads, 2) qwd_apply_kernel(const QwdApplyArgs a)
{
    const int64_t n = a.n;
    const int64_t rows = (n + kRow - 1) / kRow;
    Packed<BITS> cur;
    unsigned short cur_s = 0;
    float nref[8];   // the next row's reference, loaded one row ahead with its codes
    auto load = [&](int64_t row) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        if (e0 >= n) return;
        cur = load_codes<BITS>(a.codes, e0 >> 3);
        cur_s = __ldg(a.scales + (e0 >> a.log2B));
        const int64_t rem = n - e0;
        if (rem >= 8) {
            ld8_f32(a.ref + e0, nref);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) nref[j] = (j < rem) ? a.ref[e0 + j] : 0.0f;
        }
    };
    if ((int64_t)blockIdx.x < rows) load(blockIdx.x);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t e0 = row * kRow + (int64_t)threadIdx.x * kPiece;
        const int64_t rem = n - e0;
        const int valid = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
        float r[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = nref[j];
        uint32_t h[4];
        level_pairs<BITS>(cur, h);
        const unsigned short s = cur_s;          // this row's scale: load() below replaces cur_s
        __syncthreads();   // the CTA's next-row loads reach DRAM together (0.925 -> 0.960)
        if (row + gridDim.x < rows) load(row + gridDim.x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int jl = pair_lo<BITS>(i), jh = pair_hi<BITS>(i);
            r[jl] = fma_f16(s, (unsigned short)(h[i] & 0xFFFFu), r[jl]);   // fl(ref + s*q)
            r[jh] = fma_f16(s, (unsigned short)(h[i] >> 16), r[jh]);
        }
        if (valid == 8) {
            st8_f32(a.ref + e0, r);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) if (j < valid) a.ref[e0 + j] = r[j];
        }
        if constexpr (WOUT == 1) {
            float* w = static_cast<float*>(a.w_out);
            if (valid == 8) {
                st8_f32(w + e0, r);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) w[e0 + j] = r[j];
            }
        } else if constexpr (WOUT == 2) {
            __nv_bfloat16* w = static_cast<__nv_bfloat16*>(a.w_out);
            if (valid == 8) {
                __nv_bfloat162 p0 = __floats2bfloat162_rn(r[0], r[1]), p1 = __floats2bfloat162_rn(r[2], r[3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(r[4], r[5]), p3 = __floats2bfloat162_rn(r[6], r[7]);
                uint4 u;
                u.x = *reinterpret_cast<uint32_t*>(&p0);
                u.y = *reinterpret_cast<uint32_t*>(&p1);
                u.z = *reinterpret_cast<uint32_t*>(&p2);
                u.w = *reinterpret_cast<uint32_t*>(&p3);
                *reinterpret_cast<uint4*>(w + e0) = u;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) if (j < valid) w[e0 + j] = __float2bfloat16_rn(r[j]);
            }
        }
    }
}

// 16 elements per thread, about two rows per CTA.  The apply reads 4.5 and
// writes 4-8 bytes per element; on 1.3e9 4-bit elements in groups of 2048
// (L2 flushed) it measured 1.04-1.05 of measured HBM with bf16 weights out or
// none (the persistent 8-element kernel 0.96 / 0.92; that kernel with a grid of
// rows / 3 CTAs 0.98 / 0.94; three to eight rows per CTA 1.03-1.04; loading the
// next row one iteration ahead made no difference).
constexpr int kApply16RowsPerCta = 2;

template <int BITS, int WOUT>
__global__ void __launch_bounds__(kWideThreads) qwd_apply16_kernel(const QwdApplyArgs a)
{
    const int64_t n = a.n;
    const int64_t rows = (n + kWideRow - 1) / kWideRow;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t e0 = row * kWideRow + (int64_t)threadIdx.x * 16;
        if (e0 >= n) continue;
        const int64_t rem = n - e0;
        const Codes16<BITS> c = load_codes16<BITS>(a.codes, e0);
        const unsigned short s = __ldg(a.scales + (e0 >> a.log2B));
        float r0[8], r1[8];
        if (rem >= 16) {
            ld8_f32(a.ref + e0, r0);
            ld8_f32(a.ref + e0 + 8, r1);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                r0[j] = j < rem ? a.ref[e0 + j] : 0.0f;
                r1[j] = j + 8 < rem ? a.ref[e0 + 8 + j] : 0.0f;
            }
        }
        uint32_t h0[4], h1[4];
        level_pairs<BITS>(c.c[0], h0);
        level_pairs<BITS>(c.c[1], h1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int jl = pair_lo<BITS>(i), jh = pair_hi<BITS>(i);
            r0[jl] = fma_f16(s, (unsigned short)(h0[i] & 0xFFFFu), r0[jl]);     // fl(ref + s*q)
            r0[jh] = fma_f16(s, (unsigned short)(h0[i] >> 16), r0[jh]);
            r1[jl] = fma_f16(s, (unsigned short)(h1[i] & 0xFFFFu), r1[jl]);
            r1[jh] = fma_f16(s, (unsigned short)(h1[i] >> 16), r1[jh]);
        }
        if (rem >= 16) {
            st8_f32(a.ref + e0, r0);
            st8_f32(a.ref + e0 + 8, r1);
            if constexpr (WOUT == 1) {
                float* w = static_cast<float*>(a.w_out) + e0;
                st8_f32(w, r0);
                st8_f32(w + 8, r1);
            } else if constexpr (WOUT == 2) {
                uint32_t wv[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    wv[i] = bf16_pair(r0[2 * i], r0[2 * i + 1]);
                    wv[4 + i] = bf16_pair(r1[2 * i], r1[2 * i + 1]);
                }
                st8_b32(static_cast<uint16_t*>(a.w_out) + e0, wv);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (j < rem) {
                    const float v = j < 8 ? r0[j] : r1[j - 8];
                    a.ref[e0 + j] = v;
                    if constexpr (WOUT == 1) static_cast<float*>(a.w_out)[e0 + j] = v;
                    if constexpr (WOUT == 2)
                        static_cast<uint16_t*>(a.w_out)[e0 + j] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                }
            }
        }
    }
}

template <int IN, int BITS, bool SR>
static cudaError_t run_qwd_encode(const EncArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    // the sender moves the bytes of an error-feedback encoder; it takes that
    // encoder's spread grid (encode_impl.cuh)
    const int grid = spread_grid(qwd_encode_kernel<IN, BITS, SR>, kThreads, cap, rows, kEnc8RowsPerCta,
                                 kEncSpreadWaves);
    qwd_encode_kernel<IN, BITS, SR><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int IN>
static cudaError_t qwd_encode_bits(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    switch (bits) {
    case 2: return sr ? run_qwd_encode<IN, 2, true>(a, st) : run_qwd_encode<IN, 2, false>(a, st);
    case 4: return sr ? run_qwd_encode<IN, 4, true>(a, st) : run_qwd_encode<IN, 4, false>(a, st);
    case 8: return sr ? run_qwd_encode<IN, 8, true>(a, st) : run_qwd_encode<IN, 8, false>(a, st);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_qwd_encode(const EncArgs& a, int dtype, int bits, bool sr, cudaStream_t st)
{
    return dtype == 0 ? qwd_encode_bits<0>(a, bits, sr, st) : qwd_encode_bits<1>(a, bits, sr, st);
}

template <int BITS, int WOUT>
static cudaError_t run_qwd_apply(const QwdApplyArgs& a, cudaStream_t st)
{
    if (a.log2B >= 4 && (reinterpret_cast<uintptr_t>(a.codes) & (code16_align<BITS>() - 1)) == 0 &&
        (reinterpret_cast<uintptr_t>(a.w_out) & 31u) == 0) {        // ref: 32-byte aligned by contract
        static std::atomic<int> resident{0};
        const int64_t rows = (a.n + kWideRow - 1) / kWideRow;
        const int grid =
            spread_grid(qwd_apply16_kernel<BITS, WOUT>, kWideThreads, resident, rows, kApply16RowsPerCta, 1);
        qwd_apply16_kernel<BITS, WOUT><<<grid, kWideThreads, 0, st>>>(a);
        return cudaGetLastError();
    }
    static std::atomic<int> cap{0};
    const int64_t rows = (a.n + kRow - 1) / kRow;
    const int grid = grid_size(qwd_apply_kernel<BITS, WOUT>, cap, rows);
    qwd_apply_kernel<BITS, WOUT><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t qwd_apply_out(const QwdApplyArgs& a, int wout, cudaStream_t st)
{
    return wout == 0 ? run_qwd_apply<BITS, 0>(a, st)
                     : (wout == 1 ? run_qwd_apply<BITS, 1>(a, st) : run_qwd_apply<BITS, 2>(a, st));
}

cudaError_t launch_qwd_apply(const uint8_t* codes, const uint16_t* scales, int64_t n, int log2B,
                             float* ref, void* w_out, int wout, int bits, cudaStream_t st)
{
    QwdApplyArgs a{codes, scales, n, log2B, ref, w_out};
    switch (bits) {
    case 2: return qwd_apply_out<2>(a, wout, st);
    case 4: return qwd_apply_out<4>(a, wout, st);
    case 8: return qwd_apply_out<8>(a, wout, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace bitscom
