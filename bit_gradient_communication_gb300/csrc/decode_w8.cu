// Decoder instantiations for exactly 8 ranks (the all-reduce of one 8-GPU node).
#define DEC_KW 8
#include "decode_impl.cuh"

namespace bitscom {
cudaError_t launch_decode_w8(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    return decode_dispatch<false>(a, bits_in, bits_out, sr, st);
}
}  // namespace bitscom
