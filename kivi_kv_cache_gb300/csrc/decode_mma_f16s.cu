// decode_mma_f16s.cu -- the one-warp-per-tile fused decode at head dim 128
// over stores with fp16 scales.
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d128_f16s(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return launch_decode_mma_impl<128, true>(a, bits, gq, stream);
}

}  // namespace kivi
