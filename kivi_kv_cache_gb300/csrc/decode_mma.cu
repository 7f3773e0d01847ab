// decode_mma.cu -- the one-warp-per-tile fused decode at head dim 128 with
// fp32 scales, and the dispatch over head dims and scale storage (the other
// instantiations are compiled in decode_mma_f16s.cu, decode_mma_d64.cu,
// decode_mma_d256.cu and decode_mma_d256_f16s.cu).
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    switch (a.D) {
        case 128:
            return a.scale_f16 ? launch_decode_mma_d128_f16s(a, bits, gq, stream)
                               : launch_decode_mma_impl<128, false>(a, bits, gq, stream);
        case 64: return launch_decode_mma_d64(a, bits, gq, stream);
        case 256:
            return a.scale_f16 ? launch_decode_mma_d256_f16s(a, bits, gq, stream)
                               : launch_decode_mma_d256(a, bits, gq, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kivi
