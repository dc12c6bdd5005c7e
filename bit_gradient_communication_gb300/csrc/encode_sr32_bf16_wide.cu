// Stochastic encoder without error feedback, 32 elements per thread: bf16
// gradients, 12- and 16-bit codes.
#include "encode_sr32.cuh"

namespace bitscom {
cudaError_t launch_encode32_sr_bf16_wide(const EncArgs& a, int bits, cudaStream_t st)
{
    return encode32_sr_bits_wide<1>(a, bits, st);
}
}  // namespace bitscom
