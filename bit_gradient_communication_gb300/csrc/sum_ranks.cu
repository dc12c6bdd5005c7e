// sum_ranks.cu -- rank-ordered fp32 sum of W full-precision arrays: the local
// reduce of the hierarchical all-reduce when local communication is not
// quantised (bitscom README, "Implemented Features": hierarchical pipeline-A,
// local reduce -> inter low-bit all-reduce -> local broadcast; "Hierarchical
// All-Reduce Options": local_quantize=False keeps the local stage in full
// precision).  out[i] = fl(...fl(fl(x_0[i]) + x_1[i])... + x_{W-1}[i]), the
// ranks in order, so every implementation gets the same bits (a collective's
// own reduction order is unspecified).
//
// HBM-bound streaming kernel: a grid of 256-thread CTAs walks 8-element
// pieces (a warp's loads of one rank are 512 or 1024 contiguous bytes); a
// thread loads its piece of every rank (256-bit loads for fp32, 128-bit for
// bf16) and writes one 256-bit store.  For W = 2, 4 or 8 (sum_fixed_kernel)
// every rank's load is in flight before the first add, over a spread grid of
// one 2048-element stretch per CTA for large launches (spread_grid in
// codec.cuh: W = 8 bf16, 1.3e9 elements, 1.06 of the measured copy bandwidth
// against 0.986 on a persistent grid; two to sixteen stretches per CTA
// 1.04-1.05); other W (sum_ranks_kernel) load four ranks at a time on a
// persistent grid.  (Pieces of 16 bf16 elements, two 128-bit loads per rank 32 bytes
// apart, measured 0.58 of the copy bandwidth on the W = 8 node-local reduce of
// a 1.3e9-element gradient, against 0.835 for four ranks in flight.)
#include "codec.cuh"
#include "launch.h"

namespace bitscom {

constexpr int kSumThreads = 256;

template <int IN>
__global__ void __launch_bounds__(kSumThreads) sum_ranks_kernel(const SumArgs a)
{
    const int64_t n = a.n;
    const int64_t pieces = (n + 7) >> 3;
    const int W = a.W;
    for (int64_t pc = (int64_t)blockIdx.x * kSumThreads + threadIdx.x; pc < pieces;
         pc += (int64_t)gridDim.x * kSumThreads) {
        const int64_t e0 = pc << 3;
        float r[8];
        if (e0 + 8 <= n) {
            // four ranks' loads in flight, then their adds in rank order (rank 0
            // sets the sum)
            for (int w0 = 0; w0 < W; w0 += 4) {
                float v[4][8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (w0 + k >= W) break;
                    if constexpr (IN == 0) {
                        ld8_f32_stream(static_cast<const float*>(a.x[w0 + k]) + e0, v[k]);
                    } else {
                        bf16x8_to_f32(ld16_stream(static_cast<const uint16_t*>(a.x[w0 + k]) + e0), v[k]);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (w0 + k >= W) break;
                    if (w0 + k == 0) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) r[j] = v[k][j];
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) r[j] = __fadd_rn(r[j], v[k][j]);
                    }
                }
            }
            st8_f32(a.out + e0, r);
        } else {
            for (int64_t i = e0; i < n; ++i) {
                float s = 0.0f;
                for (int w = 0; w < W; ++w) {
                    float v;
                    if constexpr (IN == 0) {
                        v = static_cast<const float*>(a.x[w])[i];
                    } else {
                        v = __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.x[w])[i] << 16);
                    }
                    s = w == 0 ? v : __fadd_rn(s, v);
                }
                a.out[i] = s;
            }
        }
    }
}

template <int IN, int W>
__global__ void __launch_bounds__(kSumThreads) sum_fixed_kernel(const SumArgs a)
{
    const int64_t n = a.n;
    const int64_t pieces = (n + 7) >> 3;
    for (int64_t pc = (int64_t)blockIdx.x * kSumThreads + threadIdx.x; pc < pieces;
         pc += (int64_t)gridDim.x * kSumThreads) {
        const int64_t e0 = pc << 3;
        float r[8];
        if (e0 + 8 <= n) {
            // every rank's load in flight before the first add
            float v[W][8];
#pragma unroll
            for (int w = 0; w < W; ++w) {
                if constexpr (IN == 0) {
                    ld8_f32_stream(static_cast<const float*>(a.x[w]) + e0, v[w]);
                } else {
                    bf16x8_to_f32(ld16_stream(static_cast<const uint16_t*>(a.x[w]) + e0), v[w]);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = v[0][j];
#pragma unroll
            for (int w = 1; w < W; ++w) {
#pragma unroll
                for (int j = 0; j < 8; ++j) r[j] = __fadd_rn(r[j], v[w][j]);
            }
            st8_f32(a.out + e0, r);
        } else {
            for (int64_t i = e0; i < n; ++i) {
                float s = 0.0f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    float v;
                    if constexpr (IN == 0) {
                        v = static_cast<const float*>(a.x[w])[i];
                    } else {
                        v = __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.x[w])[i] << 16);
                    }
                    s = w == 0 ? v : __fadd_rn(s, v);
                }
                a.out[i] = s;
            }
        }
    }
}

// one grid-stride stretch (kSumThreads pieces) per CTA once the launch spans
// twelve waves of resident CTAs, as the encoders' spread grids
constexpr int kSumStretchesPerCta = 1;
constexpr int kSumSpreadWaves = 12;

template <int IN, int W>
static cudaError_t run_sum_fixed(const SumArgs& a, cudaStream_t st)
{
    static std::atomic<int> cap{0};
    const int64_t pieces = (a.n + 7) >> 3;
    const int64_t blocks = (pieces + kSumThreads - 1) / kSumThreads;
    const int grid = spread_grid(sum_fixed_kernel<IN, W>, kSumThreads, cap, blocks, kSumStretchesPerCta,
                                 kSumSpreadWaves);
    sum_fixed_kernel<IN, W><<<grid, kSumThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int IN>
static cudaError_t run_sum(const SumArgs& a, cudaStream_t st)
{
    switch (a.W) {
    case 2: return run_sum_fixed<IN, 2>(a, st);
    case 4: return run_sum_fixed<IN, 4>(a, st);
    case 8: return run_sum_fixed<IN, 8>(a, st);
    default: break;
    }
    static std::atomic<int> cap{0};
    int c = cap.load(std::memory_order_relaxed);
    if (c == 0) {
        int dev = 0, occ = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sum_ranks_kernel<IN>, kSumThreads, 0);
        c = (sms > 0 ? sms : 1) * (occ > 0 ? occ : 1);
        cap.store(c, std::memory_order_relaxed);
    }
    const int64_t pieces = (a.n + 7) >> 3;
    const int64_t blocks = (pieces + kSumThreads - 1) / kSumThreads;
    const int grid = (int)(blocks < c ? blocks : c);
    sum_ranks_kernel<IN><<<grid, kSumThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_sum_ranks(const SumArgs& a, int dtype, cudaStream_t st)
{
    return dtype == 0 ? run_sum<0>(a, st) : run_sum<1>(a, st);
}

}  // namespace bitscom
