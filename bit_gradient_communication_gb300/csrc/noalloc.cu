// noalloc.cu -- bitscom_roundtrip_noalloc: quantise-then-dequantise without
// caller-provided scratch.  The intermediate codes and fp16 scales live in a
// fixed device array defined in this file, so neither the library nor the
// caller allocates anything for the call.
//
// Why it exists: some callers cannot allocate device memory at the point
// where they want to simulate quantisation -- for instance a gradient hook
// that only receives the gradient buffer and must not call the CUDA allocator
// (cudaMalloc / cudaFree can synchronise the device and compete with the
// framework's caching allocator, which may already hold all free memory).
//
// Limits and sharing rules (also stated in include/bitscom.h):
//   * capacity: 8 MiB of codes + 1 MiB of scales per device.  The first call
//     on a device looks the array's address up; with CUDA's lazy module
//     loading that lookup loads this file's module, which reserves the array
//     (and may synchronise the device), so callers make that call at set-up
//     time.  The array stays until the process exits;
//   * the address is cached per device number; after cudaDeviceReset the
//     cached address is stale and calls on that device are not supported;
//   * one array per device, shared by every call on that device: calls whose
//     kernels overlap on the GPU (different streams, or different host threads
//     without ordering) race on it;
//   * the array keeps the last call's contents; nothing in it needs to start at
//     zero because the encoder writes every code byte (padding included) and
//     every scale before the decoder reads them.
#include "bitscom.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launch.h"

constexpr int64_t kCodeBytes = 8ll << 20;    // codes region
constexpr int64_t kScaleBytes = 1ll << 20;   // fp16 scales region
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_roundtrip_scratch[kCodeBytes + kScaleBytes];

namespace {

// Device address of g_roundtrip_scratch, looked up once per device with that
// device current.  In host code the symbol is only a host-side stand-in.
std::mutex g_mutex;
void* g_scratch[kMaxDevices] = {};

bitscom_status scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        bitscom::record_cuda_error(e);
        return BITSCOM_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return BITSCOM_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_roundtrip_scratch);
        if (e != cudaSuccess || !p) {
            bitscom::record_cuda_error(e);
            return BITSCOM_ECUDA;
        }
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return BITSCOM_OK;
}

}  // namespace

extern "C" {

int64_t bitscom_roundtrip_noalloc_max_elements(int32_t bits, int32_t block)
{
    if (block < 8 || block > 4096 || (block & (block - 1)) != 0 ||
        !(bits == 1 || bits == 2 || bits == 4 || bits == 8 || bits == 12 || bits == 16))
        return -1;
    // whole blocks whose codes fit the codes region and whose scales fit the scales region
    const int64_t by_codes = kCodeBytes / ((int64_t)block * bits / 8);
    const int64_t by_scales = kScaleBytes / 2;
    const int64_t blocks = by_codes < by_scales ? by_codes : by_scales;
    return blocks * block;
}

bitscom_status bitscom_roundtrip_noalloc(const void* x, bitscom_dtype dt, int64_t n, float* err,
                                         const bitscom_qparams* p, float* deq_out, void* cuda_stream)
{
    if (!p) return BITSCOM_EINVAL;
    const int64_t cap = bitscom_roundtrip_noalloc_max_elements(p->bits, p->block);
    if (cap < 0 || n < 0) return BITSCOM_EINVAL;
    if (n > cap) return BITSCOM_EINVAL;   // beyond the fixed scratch capacity
    if (n == 0) return BITSCOM_OK;
    void* base = nullptr;
    const bitscom_status st = scratch_address(&base);
    if (st != BITSCOM_OK) return st;
    unsigned char* codes = static_cast<unsigned char*>(base);
    uint16_t* scales = reinterpret_cast<uint16_t*>(codes + kCodeBytes);
    return bitscom_roundtrip(x, dt, n, err, p, codes, scales, deq_out, cuda_stream);
}

}  // extern "C"
