// Decoder instantiations for 1..7 ranks (rank count read at run time).
#define DEC_KW 0
#include "decode_impl.cuh"

namespace bitscom {
cudaError_t launch_decode_few(const DecArgs& a, int bits_in, int bits_out, bool sr, cudaStream_t st)
{
    return decode_dispatch<false>(a, bits_in, bits_out, sr, st);
}
}  // namespace bitscom
