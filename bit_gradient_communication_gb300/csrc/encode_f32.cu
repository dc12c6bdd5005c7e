// Encoder instantiations for fp32 gradients.
#include "encode_impl.cuh"

namespace bitscom {
cudaError_t launch_encode_f32(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    return encode_dispatch<0>(a, bits, sr, st);
}

cudaError_t launch_roundtrip_f32(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    return roundtrip_dispatch<0>(a, bits, sr, st);
}
}  // namespace bitscom
