// Stochastic encoder without error feedback, 32 elements per thread: f32
// gradients, 2-, 4- and 8-bit codes.
#include "encode_sr32.cuh"

namespace bitscom {
cudaError_t launch_encode32_sr_f32(const EncArgs& a, int bits, cudaStream_t st)
{
    return encode32_sr_bits_narrow<0>(a, bits, st);
}
}  // namespace bitscom
