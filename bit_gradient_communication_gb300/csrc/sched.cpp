// sched.cpp -- host bucket scheduler: fusion buckets (25 MB in the ACP-SGD and
// DeAR READMEs) issued round-robin on the scheduler's own CUDA streams, with
// one fork event on the caller's stream and one join event per used stream
// (bitscom README, "Implemented Features": dual-stream scheduling).
#include "bitscom.h"

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <chrono>
#include <cstdint>
#include <thread>
#include <vector>

#include "launch.h"

struct bitscom_sched {
    int n_streams = 0;
    int64_t bucket_bytes = 0;
    int device = 0;
    cudaStream_t streams[8] = {};
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[8] = {};
};

namespace {

constexpr int kMaxStreams = 8;

// NVTX range over a scope of host-side issue (header-only NVTX3: nearly free
// unless a profiler is attached), so a trace shows which bucket and phase
// issued which launches.
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

int64_t plan_unit(int32_t block) { return block > 128 ? block : 128; }

// Elements per bucket (0 = the whole call is one bucket).
int64_t bucket_elems(int64_t bucket_bytes, int32_t elem_bytes, int64_t unit)
{
    if (bucket_bytes <= 0) return 0;
    int64_t per = bucket_bytes / elem_bytes / unit * unit;
    return per < unit ? unit : per;
}

bitscom_status err_of(cudaError_t e)
{
    if (e == cudaSuccess) return BITSCOM_OK;
    bitscom::record_cuda_error(e);
    return BITSCOM_ECUDA;
}

// Order the scheduler's streams after everything already on `caller`.
bitscom_status fork(bitscom_sched* s, cudaStream_t caller, int used)
{
    bitscom_status st = err_of(cudaEventRecord(s->fork, caller));
    for (int i = 0; st == BITSCOM_OK && i < used; ++i)
        st = err_of(cudaStreamWaitEvent(s->streams[i], s->fork, 0));
    return st;
}

// Order later work on `caller` after every bucket.
bitscom_status join(bitscom_sched* s, cudaStream_t caller, int used)
{
    bitscom_status st = BITSCOM_OK;
    for (int i = 0; st == BITSCOM_OK && i < used; ++i) {
        st = err_of(cudaEventRecord(s->join[i], s->streams[i]));
        if (st == BITSCOM_OK) st = err_of(cudaStreamWaitEvent(caller, s->join[i], 0));
    }
    return st;
}

int64_t offset_bytes(int64_t elems, int bits) { return elems * bits / 8; }

}  // namespace

extern "C" {

bitscom_status bitscom_sched_create(int32_t n_streams, int64_t bucket_bytes, bitscom_sched** out)
{
    if (!out || n_streams < 1 || n_streams > kMaxStreams) return BITSCOM_EINVAL;
    *out = nullptr;
    bitscom_sched* s = new bitscom_sched;
    s->n_streams = n_streams;
    s->bucket_bytes = bucket_bytes;
    bitscom_status st = err_of(cudaGetDevice(&s->device));
    if (st == BITSCOM_OK) st = err_of(cudaEventCreateWithFlags(&s->fork, cudaEventDisableTiming));
    for (int i = 0; st == BITSCOM_OK && i < n_streams; ++i) {
        st = err_of(cudaStreamCreateWithFlags(&s->streams[i], cudaStreamNonBlocking));
        if (st == BITSCOM_OK) st = err_of(cudaEventCreateWithFlags(&s->join[i], cudaEventDisableTiming));
    }
    if (st != BITSCOM_OK) {
        bitscom_sched_destroy(s);
        return st;
    }
    *out = s;
    return BITSCOM_OK;
}

bitscom_status bitscom_sched_destroy(bitscom_sched* s)
{
    if (!s) return BITSCOM_EINVAL;
    for (int i = 0; i < kMaxStreams; ++i) {
        if (s->streams[i]) cudaStreamSynchronize(s->streams[i]);
        if (s->join[i]) cudaEventDestroy(s->join[i]);
        if (s->streams[i]) cudaStreamDestroy(s->streams[i]);
    }
    if (s->fork) cudaEventDestroy(s->fork);
    delete s;
    return BITSCOM_OK;
}

int64_t bitscom_sched_plan(int64_t n, int32_t elem_bytes, int32_t block, int64_t bucket_bytes,
                           int64_t* starts, int64_t cap)
{
    if (n < 0 || (elem_bytes != 2 && elem_bytes != 4) || block < 8 || block > 4096 ||
        (block & (block - 1)) != 0 || (starts && cap < 0))
        return -1;
    if (n == 0) {
        if (starts && cap >= 0) starts[0] = 0;
        return 0;
    }
    const int64_t per = bucket_elems(bucket_bytes, elem_bytes, plan_unit(block));
    const int64_t count = per == 0 ? 1 : (n + per - 1) / per;
    if (starts) {
        for (int64_t k = 0; k <= count && k <= cap; ++k) {
            const int64_t e = per == 0 ? (k == 0 ? 0 : n) : k * per;
            starts[k] = e < n ? e : n;
        }
    }
    return count;
}

bitscom_status bitscom_sched_quantize_pack(bitscom_sched* s, const void* x, bitscom_dtype dt,
                                           int64_t n, float* err, const bitscom_qparams* p,
                                           void* codes_out, uint16_t* scales_out, void* cuda_stream)
{
    if (!s) return BITSCOM_EINVAL;
    bitscom_status st = bitscom::check_encode(x, dt, n, err, p, codes_out, scales_out);
    if (st != BITSCOM_OK || n == 0) return st;
    const int esz = dt == BITSCOM_F32 ? 4 : 2;
    const int64_t per = bucket_elems(s->bucket_bytes, esz, plan_unit(p->block));
    const int64_t count = per == 0 ? 1 : (n + per - 1) / per;
    const int used = count < s->n_streams ? (int)count : s->n_streams;
    cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);
    Range whole("bitscom.sched.quantize_pack");
    st = fork(s, caller, used);
    for (int64_t k = 0; st == BITSCOM_OK && k < count; ++k) {
        Range bucket("bitscom.bucket");
        const int64_t b0 = per == 0 ? 0 : k * per;
        const int64_t nb = per == 0 ? n : (n - b0 < per ? n - b0 : per);
        bitscom_qparams q = *p;
        q.index_offset = p->index_offset + (uint64_t)b0;
        st = bitscom_quantize_pack(static_cast<const char*>(x) + b0 * esz, dt, nb, err ? err + b0 : nullptr,
                                   &q, static_cast<char*>(codes_out) + offset_bytes(b0, p->bits),
                                   scales_out + b0 / p->block, s->streams[k % s->n_streams]);
    }
    const bitscom_status jst = join(s, caller, used);
    return st != BITSCOM_OK ? st : jst;
}

bitscom_status bitscom_sched_allreduce(bitscom_sched* s, int32_t W, const void* const* x,
                                       bitscom_dtype dt, int64_t n, float* const* err,
                                       const bitscom_qparams* p1, void* const* codes,
                                       uint16_t* const* scales, const bitscom_qparams* p2,
                                       float* err2, void* codes_out, uint16_t* scales_out,
                                       float* sum_out, void* cuda_stream)
{
    if (!s || !x || !p1 || !codes || !scales || W < 1 || W > bitscom::kMaxRanks || n < 0)
        return BITSCOM_EINVAL;
    // every rank uses one code format
    for (int w = 1; w < W; ++w)
        if (p1[w].bits != p1[0].bits || p1[w].block != p1[0].block) return BITSCOM_EINVAL;
    for (int w = 0; w < W; ++w) {
        const bitscom_status st = bitscom::check_encode(x[w], dt, n, err ? err[w] : nullptr, &p1[w],
                                                        codes[w], scales[w]);
        if (st != BITSCOM_OK) return st;
    }
    {
        std::vector<const void*> ci(codes, codes + W);
        std::vector<const uint16_t*> si(scales, scales + W);
        const bitscom_status st = bitscom::check_decode(ci.data(), si.data(), W, n, &p1[0], sum_out,
                                                        err2, p2, codes_out, scales_out);
        if (st != BITSCOM_OK) return st;
    }
    if (p2 && p2->block != p1[0].block && (p2->block % p1[0].block) != 0 && (p1[0].block % p2->block) != 0)
        return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;

    const int esz = dt == BITSCOM_F32 ? 4 : 2;
    const int32_t B1 = p1[0].block, B2 = p2 ? p2->block : B1;
    const int64_t U = B1 > B2 ? B1 : B2;                 // chunk / bucket alignment unit
    const int64_t per = bucket_elems(s->bucket_bytes, esz, U > 128 ? U : 128);
    const int64_t count = per == 0 ? 1 : (n + per - 1) / per;
    const int used = count < s->n_streams ? (int)count : s->n_streams;
    cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);
    Range whole("bitscom.sched.allreduce");
    bitscom_status st = fork(s, caller, used);
    std::vector<const void*> cin(W);
    std::vector<const uint16_t*> sin(W);
    for (int64_t k = 0; st == BITSCOM_OK && k < count; ++k) {
        cudaStream_t str = s->streams[k % s->n_streams];
        const int64_t b0 = per == 0 ? 0 : k * per;
        const int64_t nbk = per == 0 ? n : (n - b0 < per ? n - b0 : per);
        // stage 1 on every rank
        {
            Range enc("bitscom.bucket.encode");
            for (int w = 0; st == BITSCOM_OK && w < W; ++w) {
                bitscom_qparams q = p1[w];
                q.index_offset = p1[w].index_offset + (uint64_t)b0;
                st = bitscom_quantize_pack(static_cast<const char*>(x[w]) + b0 * esz, dt, nbk,
                                           (err && err[w]) ? err[w] + b0 : nullptr, &q,
                                           static_cast<char*>(codes[w]) + offset_bytes(b0, p1[w].bits),
                                           scales[w] + b0 / B1, str);
            }
        }
        // all-to-all by pointer arithmetic: chunk c = units [c*cu, (c+1)*cu)
        Range dec("bitscom.bucket.decode");
        const int64_t units = (nbk + U - 1) / U;
        const int64_t cu = (units + W - 1) / W;
        for (int c = 0; st == BITSCOM_OK && c < W; ++c) {
            const int64_t u0 = (int64_t)c * cu;
            if (u0 >= units) break;
            const int64_t lo = b0 + u0 * U;
            const int64_t hi_local = (u0 + cu) * U < nbk ? (u0 + cu) * U : nbk;
            const int64_t nc = b0 + hi_local - lo;
            for (int w = 0; w < W; ++w) {
                cin[w] = static_cast<const char*>(codes[w]) + offset_bytes(lo, p1[0].bits);
                sin[w] = scales[w] + lo / B1;
            }
            bitscom_qparams q2;
            if (p2) {
                q2 = *p2;
                q2.index_offset = p2->index_offset + (uint64_t)lo;
            }
            st = bitscom_unpack_dequant_reduce_requant(
                cin.data(), sin.data(), W, nc, &p1[0], sum_out ? sum_out + lo : nullptr,
                err2 ? err2 + lo : nullptr, p2 ? &q2 : nullptr,
                p2 ? static_cast<char*>(codes_out) + offset_bytes(lo, p2->bits) : nullptr,
                p2 ? scales_out + lo / B2 : nullptr, str);
        }
    }
    const bitscom_status jst = join(s, caller, used);
    return st != BITSCOM_OK ? st : jst;
}

bitscom_status bitscom_sched_wait(bitscom_sched* s, void* cuda_stream, double timeout_s)
{
    if (!s || timeout_s < 0) return BITSCOM_EINVAL;
    const auto deadline = std::chrono::steady_clock::now() +
                          std::chrono::duration_cast<std::chrono::steady_clock::duration>(
                              std::chrono::duration<double>(timeout_s));
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    for (;;) {
        const cudaError_t e = cudaStreamQuery(st);
        if (e == cudaSuccess) return BITSCOM_OK;
        if (e != cudaErrorNotReady) return err_of(e);
        if (std::chrono::steady_clock::now() >= deadline) return BITSCOM_ETIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

}  // extern "C"
