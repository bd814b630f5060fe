// Decode attention over a cache whose tokens are Walsh-Hadamard rotated
// before quantization, contiguous layout: the kernels of decode_kernel.cuh
// instantiated with the query rotation, the two-part value weights and the
// back-rotation in the merge.  A translation unit of its own so that the
// instantiation sets compile in parallel.
#include "decode_kernel.cuh"

namespace kvq {

cudaError_t launch_rot(const DecodeArgs &a, int gq, cudaStream_t stream) {
  return a.geo.bits == 2 ? launch_b<2, false, true, false>(a, gq, stream) : launch_b<4, false, true, false>(a, gq, stream);
}

}  // namespace kvq
