// Decode attention over a block-paged cache whose tokens are Walsh-Hadamard
// rotated before quantization (decode_rot.cu with the block-table fetch).
#include "decode_kernel.cuh"

namespace kvq {

cudaError_t launch_rot_paged(const DecodeArgs &a, int gq, cudaStream_t stream) {
  return a.geo.bits == 2 ? launch_b<2, true, true, false>(a, gq, stream) : launch_b<4, true, true, false>(a, gq, stream);
}

}  // namespace kvq
