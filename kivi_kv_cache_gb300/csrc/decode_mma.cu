// decode_mma.cu -- the one-warp-per-tile fused decode at head dim 128, and the
// dispatch over head dims (64 and 256 are compiled in decode_mma_d64.cu and
// decode_mma_d256.cu).
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    switch (a.D) {
        case 128: return launch_decode_mma_impl<128>(a, bits, gq, stream);
        case 64: return launch_decode_mma_d64(a, bits, gq, stream);
        case 256: return launch_decode_mma_d256(a, bits, gq, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kivi
