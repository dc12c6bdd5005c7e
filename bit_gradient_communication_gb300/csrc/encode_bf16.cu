// Encoder instantiations for bf16 gradients.
#include "encode_impl.cuh"

namespace bitscom {
cudaError_t launch_encode_bf16(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    return encode_dispatch<1>(a, bits, sr, st);
}

cudaError_t launch_roundtrip_bf16(const EncArgs& a, int bits, bool sr, cudaStream_t st)
{
    return roundtrip_dispatch<1>(a, bits, sr, st);
}
}  // namespace bitscom
