// api.cpp -- the C ABI entry points of include/bitscom.h: host-side argument
// checks (nothing is enqueued on a bad argument), then one kernel launch each.
#include "bitscom.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "launch.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

bitscom_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return BITSCOM_OK;
    if (e == cudaErrorNotSupported) return BITSCOM_EUNSUPPORTED;
    std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
    return BITSCOM_ECUDA;
}

bool valid_bits(int b) { return b == 1 || b == 2 || b == 4 || b == 8 || b == 12 || b == 16; }

int log2_block(int B)
{
    if (B < 8 || B > 4096 || (B & (B - 1)) != 0) return -1;
    int l = 0;
    while ((1 << l) < B) ++l;
    return l;
}

bool valid_hadamard(int H, int B)
{
    return H == 0 || (H >= 8 && H <= 256 && (H & (H - 1)) == 0 && B % H == 0);
}

bool valid_params(const bitscom_qparams* p)
{
    return p && valid_bits(p->bits) && log2_block(p->block) >= 0 &&
           (p->rounding == BITSCOM_RTN || p->rounding == BITSCOM_SR) &&
           valid_hadamard(p->hadamard, p->block) && p->reserved == 0;
}

// The Walsh-Hadamard rotation needs whole transform blocks and has kernels
// for 2-, 4- and 8-bit codes.
bitscom_status check_hadamard(const bitscom_qparams* p, int64_t n)
{
    if (!p->hadamard) return BITSCOM_OK;
    if (n % p->hadamard != 0) return BITSCOM_EINVAL;
    if (p->bits != 2 && p->bits != 4 && p->bits != 8) return BITSCOM_EUNSUPPORTED;
    return BITSCOM_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Width of one thread's code store/load: 8 codes = b bytes.
uintptr_t code_align(int bits)
{
    switch (bits) {
    case 1: return 1;
    case 2: return 2;
    case 4: return 4;
    case 8: return 8;
    case 12: return 4;
    default: return 16;
    }
}

}  // namespace

namespace bitscom {

bitscom_status check_encode(const void* x, bitscom_dtype dt, int64_t n, const float* err,
                            const bitscom_qparams* p, const void* codes, const uint16_t* scales)
{
    if (!valid_params(p) || n < 0 || (dt != BITSCOM_F32 && dt != BITSCOM_BF16)) return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;
    if (!x || !codes || !scales) return BITSCOM_EINVAL;
    const bitscom_status h = check_hadamard(p, n);
    if (h != BITSCOM_OK) return h;
    if (!aligned(x, dt == BITSCOM_F32 ? 32 : 16) || (err && !aligned(err, 32)) ||
        !aligned(codes, code_align(p->bits)) || !aligned(scales, 2))
        return BITSCOM_EALIGN;
    return BITSCOM_OK;
}

bitscom_status check_decode(const void* const* codes_in, const uint16_t* const* scales_in, int32_t W,
                            int64_t n, const bitscom_qparams* p_in, const float* sum_out,
                            const float* err2, const bitscom_qparams* p_out, const void* codes_out,
                            const uint16_t* scales_out)
{
    if (!valid_params(p_in) || n < 0 || W < 1 || W > kMaxRanks) return BITSCOM_EINVAL;
    if (p_out && !valid_params(p_out)) return BITSCOM_EINVAL;
    if (p_out && p_out->hadamard != p_in->hadamard) return BITSCOM_EINVAL;   // one rotated domain
    if (err2 && !p_out) return BITSCOM_EINVAL;
    if (!sum_out && !p_out) return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;
    if (!codes_in || !scales_in) return BITSCOM_EINVAL;
    if (p_out && (!codes_out || !scales_out)) return BITSCOM_EINVAL;
    for (int w = 0; w < W; ++w) {
        if (!codes_in[w] || !scales_in[w]) return BITSCOM_EINVAL;
        if (!aligned(codes_in[w], code_align(p_in->bits)) || !aligned(scales_in[w], 2)) return BITSCOM_EALIGN;
    }
    if ((sum_out && !aligned(sum_out, 32)) || (err2 && !aligned(err2, 32))) return BITSCOM_EALIGN;
    if (p_out && (!aligned(codes_out, code_align(p_out->bits)) || !aligned(scales_out, 2))) return BITSCOM_EALIGN;
    return BITSCOM_OK;
}

const char* record_cuda_error(cudaError_t e)
{
    std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
    return g_last_cuda_error;
}

}  // namespace bitscom

extern "C" {

int64_t bitscom_num_blocks(int64_t n, int32_t block)
{
    if (n < 0 || block <= 0) return -1;
    return (n + block - 1) / block;
}

int64_t bitscom_packed_bytes(int64_t n, int32_t bits, int32_t block)
{
    if (n < 0 || block <= 0 || !valid_bits(bits)) return -1;
    return (n + block - 1) / block * block * bits / 8;
}

const char* bitscom_status_string(bitscom_status s)
{
    switch (s) {
    case BITSCOM_OK: return "ok";
    case BITSCOM_EINVAL: return "invalid argument";
    case BITSCOM_EALIGN: return "pointer not aligned";
    case BITSCOM_EUNSUPPORTED: return "unsupported combination";
    case BITSCOM_ECUDA: return "CUDA error";
    case BITSCOM_ETIMEOUT: return "timed out";
    default: return "unknown status";
    }
}

const char* bitscom_last_cuda_error(void) { return g_last_cuda_error; }

bitscom_status bitscom_quantize_pack(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                     const bitscom_qparams* p, void* codes_out,
                                     uint16_t* scales_out, void* cuda_stream)
{
    const bitscom_status chk = bitscom::check_encode(x, dt, n, err, p, codes_out, scales_out);
    if (chk != BITSCOM_OK || n == 0) return chk;
    bitscom::EncArgs a;
    a.x = x;
    a.err = err;
    a.n = n;
    a.log2B = log2_block(p->block);
    a.nb = (n + p->block - 1) / p->block;
    a.codes = static_cast<uint8_t*>(codes_out);
    a.scales = scales_out;
    a.keys = bitscom::philox_keys(p->seed, p->philox_stream);
    a.index_offset = p->index_offset;
    a.hadamard = p->hadamard;
    return cuda_status(bitscom::launch_encode(a, dt == BITSCOM_F32 ? 0 : 1, p->bits,
                                              p->rounding == BITSCOM_SR,
                                              static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_unpack_dequant_reduce_requant(
    const void* const* codes_in, const uint16_t* const* scales_in, int32_t W, int64_t n,
    const bitscom_qparams* p_in, float* sum_out, float* err2, const bitscom_qparams* p_out,
    void* codes_out, uint16_t* scales_out, void* cuda_stream)
{
    const bitscom_status chk = bitscom::check_decode(codes_in, scales_in, W, n, p_in, sum_out, err2,
                                                     p_out, codes_out, scales_out);
    if (chk != BITSCOM_OK || n == 0) return chk;
    if (W == 1 && !p_out && p_in->hadamard == 0) {
        // one rank, no requantisation: the sum is fl(s*q) itself, which the
        // all-gather-side decode kernel writes with mul = 1 (fl(d * 1) = d)
        bitscom::DqArgs d;
        d.codes = static_cast<const uint8_t*>(codes_in[0]);
        d.scales = scales_in[0];
        d.n = n;
        d.log2B = log2_block(p_in->block);
        d.mul = 1.0f;
        d.out = sum_out;
        d.hadamard = 0;
        return cuda_status(bitscom::launch_dequant(d, p_in->bits, 0, static_cast<cudaStream_t>(cuda_stream)));
    }
    bitscom::DecArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int w = 0; w < W; ++w) {
        a.codes[w] = static_cast<const uint8_t*>(codes_in[w]);
        a.scales[w] = scales_in[w];
    }
    a.W = W;
    a.n = n;
    a.log2Bin = log2_block(p_in->block);
    a.log2Bout = p_out ? log2_block(p_out->block) : a.log2Bin;
    a.nb_out = p_out ? (n + p_out->block - 1) / p_out->block : 0;
    a.sum_out = sum_out;
    a.err2 = err2;
    a.codes_out = static_cast<uint8_t*>(codes_out);
    a.scales_out = scales_out;
    if (p_out) {
        a.keys = bitscom::philox_keys(p_out->seed, p_out->philox_stream);
        a.index_offset = p_out->index_offset;
    }
    return cuda_status(bitscom::launch_decode(a, p_in->bits, p_out ? p_out->bits : 0,
                                              p_out && p_out->rounding == BITSCOM_SR,
                                              static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_unpack_dequant(const void* codes, const uint16_t* scales, int64_t n,
                                     const bitscom_qparams* p, float mul, bitscom_dtype out_dt,
                                     void* out, void* cuda_stream)
{
    if (!valid_params(p) || n < 0 || (out_dt != BITSCOM_F32 && out_dt != BITSCOM_BF16)) return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;
    if (!codes || !scales || !out) return BITSCOM_EINVAL;
    const bitscom_status h = check_hadamard(p, n);
    if (h != BITSCOM_OK) return h;
    if (!aligned(codes, code_align(p->bits)) || !aligned(scales, 2) ||
        !aligned(out, out_dt == BITSCOM_F32 ? 32 : 16))
        return BITSCOM_EALIGN;
    bitscom::DqArgs a;
    a.codes = static_cast<const uint8_t*>(codes);
    a.scales = scales;
    a.n = n;
    a.log2B = log2_block(p->block);
    a.mul = mul;
    a.out = out;
    a.hadamard = p->hadamard;
    return cuda_status(bitscom::launch_dequant(a, p->bits, out_dt == BITSCOM_F32 ? 0 : 1,
                                               static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_sum_ranks(const void* const* x, bitscom_dtype dt, int32_t W, int64_t n, float* out,
                                 void* cuda_stream)
{
    if (W < 1 || W > bitscom::kMaxRanks || n < 0 || (dt != BITSCOM_F32 && dt != BITSCOM_BF16)) return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;
    if (!x || !out) return BITSCOM_EINVAL;
    bitscom::SumArgs a;
    for (int w = 0; w < W; ++w) {
        if (!x[w]) return BITSCOM_EINVAL;
        if (!aligned(x[w], dt == BITSCOM_F32 ? 32 : 16)) return BITSCOM_EALIGN;
        a.x[w] = x[w];
    }
    if (!aligned(out, 32)) return BITSCOM_EALIGN;
    a.W = W;
    a.n = n;
    a.out = out;
    return cuda_status(bitscom::launch_sum_ranks(a, dt == BITSCOM_F32 ? 0 : 1, static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_qwd_encode(const void* w, bitscom_dtype dt, int64_t n, float* ref,
                                  const bitscom_qparams* p, void* codes_out, uint16_t* scales_out,
                                  void* cuda_stream)
{
    if (!ref && n > 0) return BITSCOM_EINVAL;
    if (p && p->hadamard) return BITSCOM_EINVAL;
    const bitscom_status chk = bitscom::check_encode(w, dt, n, ref, p, codes_out, scales_out);
    if (chk != BITSCOM_OK || n == 0) return chk;
    if (p->bits != 2 && p->bits != 4 && p->bits != 8) return BITSCOM_EUNSUPPORTED;
    bitscom::EncArgs a;
    a.x = w;
    a.err = ref;
    a.n = n;
    a.log2B = log2_block(p->block);
    a.nb = (n + p->block - 1) / p->block;
    a.codes = static_cast<uint8_t*>(codes_out);
    a.scales = scales_out;
    a.keys = bitscom::philox_keys(p->seed, p->philox_stream);
    a.index_offset = p->index_offset;
    a.hadamard = 0;
    return cuda_status(bitscom::launch_qwd_encode(a, dt == BITSCOM_F32 ? 0 : 1, p->bits,
                                                  p->rounding == BITSCOM_SR,
                                                  static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_qwd_apply(const void* codes, const uint16_t* scales, int64_t n,
                                 const bitscom_qparams* p, float* ref, void* w_out,
                                 bitscom_dtype w_dt, void* cuda_stream)
{
    if (!valid_params(p) || p->hadamard || n < 0 || (w_dt != BITSCOM_F32 && w_dt != BITSCOM_BF16))
        return BITSCOM_EINVAL;
    if (n == 0) return BITSCOM_OK;
    if (!codes || !scales || !ref) return BITSCOM_EINVAL;
    if (!aligned(codes, code_align(p->bits)) || !aligned(scales, 2) || !aligned(ref, 32) ||
        (w_out && !aligned(w_out, w_dt == BITSCOM_F32 ? 32 : 16)))
        return BITSCOM_EALIGN;
    if (p->bits != 2 && p->bits != 4 && p->bits != 8) return BITSCOM_EUNSUPPORTED;
    const int wout = w_out == nullptr ? 0 : (w_dt == BITSCOM_F32 ? 1 : 2);
    return cuda_status(bitscom::launch_qwd_apply(static_cast<const uint8_t*>(codes), scales, n,
                                                 log2_block(p->block), ref, w_out, wout, p->bits,
                                                 static_cast<cudaStream_t>(cuda_stream)));
}

bitscom_status bitscom_roundtrip(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                 const bitscom_qparams* p, void* codes_tmp,
                                 uint16_t* scales_tmp, float* deq_out, void* cuda_stream)
{
    if (n > 0 && !deq_out) return BITSCOM_EINVAL;
    if (deq_out && !aligned(deq_out, 32)) return BITSCOM_EALIGN;
    if (!err && p && p->hadamard == 0 && n > 0) {
        // one pass: codes, scales and fl(s*q) from the same registers
        const bitscom_status chk = bitscom::check_encode(x, dt, n, err, p, codes_tmp, scales_tmp);
        if (chk != BITSCOM_OK) return chk;
        bitscom::EncArgs a;
        a.x = x;
        a.err = nullptr;
        a.n = n;
        a.log2B = log2_block(p->block);
        a.nb = (n + p->block - 1) / p->block;
        a.codes = static_cast<uint8_t*>(codes_tmp);
        a.scales = scales_tmp;
        a.keys = bitscom::philox_keys(p->seed, p->philox_stream);
        a.index_offset = p->index_offset;
        a.hadamard = 0;
        a.deq = deq_out;
        const cudaError_t e = bitscom::launch_roundtrip(a, dt == BITSCOM_F32 ? 0 : 1, p->bits,
                                                        p->rounding == BITSCOM_SR,
                                                        static_cast<cudaStream_t>(cuda_stream));
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    bitscom_status s = bitscom_quantize_pack(x, dt, n, err, p, codes_tmp, scales_tmp, cuda_stream);
    if (s != BITSCOM_OK || n == 0) return s;
    return bitscom_unpack_dequant(codes_tmp, scales_tmp, n, p, 1.0f, BITSCOM_F32, deq_out, cuda_stream);
}

}  // extern "C"
