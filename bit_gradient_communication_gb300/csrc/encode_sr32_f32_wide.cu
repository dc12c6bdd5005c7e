// Stochastic encoder without error feedback, 32 elements per thread: f32
// gradients, 12- and 16-bit codes.
#include "encode_sr32.cuh"

namespace bitscom {
cudaError_t launch_encode32_sr_f32_wide(const EncArgs& a, int bits, cudaStream_t st)
{
    return encode32_sr_bits_wide<0>(a, bits, st);
}
}  // namespace bitscom
