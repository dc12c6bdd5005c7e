// Decoder instantiations for W > 8 ranks (groups of 8 ranks per pass).
#define DEC_KW 0
#include "decode_impl.cuh"

namespace bitscom {
cudaError_t launch_decode_many(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    return decode_dispatch<true>(a, bits_in, bits_out, sr, st);
}
}  // namespace bitscom
