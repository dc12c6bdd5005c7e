// Stochastic encoder without error feedback, 32 elements per thread: bf16
// gradients, 2-, 4- and 8-bit codes.
#include "encode_sr32.cuh"

namespace bitscom {
cudaError_t launch_encode32_sr_bf16(const EncArgs& a, int bits, cudaStream_t st)
{
    return encode32_sr_bits_narrow<1>(a, bits, st);
}
}  // namespace bitscom
