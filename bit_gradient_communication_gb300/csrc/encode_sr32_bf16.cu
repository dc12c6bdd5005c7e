// Stochastic encoder without error feedback, 32 elements per thread, for bf16 gradients.
#include "encode_sr32.cuh"

namespace bitscom {
cudaError_t launch_encode32_sr_bf16(const EncArgs& a, int bits, cudaStream_t st)
{
    return encode32_sr_bits<1>(a, bits, st);
}
}  // namespace bitscom
