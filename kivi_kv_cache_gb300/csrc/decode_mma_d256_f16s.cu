// decode_mma_d256_f16s.cu -- the one-warp-per-tile fused decode at head dim
// 256 over stores with fp16 scales.
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d256_f16s(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return launch_decode_mma_impl<256, true>(a, bits, gq, stream);
}

}  // namespace kivi
