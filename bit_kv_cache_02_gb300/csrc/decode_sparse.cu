// Decode attention over dense-and-sparse blocks (each slice's largest
// element kept as an fp16 entry), contiguous layout: the kernels of
// decode_kernel.cuh instantiated with the outlier corrections of the scores
// and the values.  A translation unit of its own so that the instantiation
// sets compile in parallel.
#include "decode_kernel.cuh"

namespace kvq {

cudaError_t launch_sparse(const DecodeArgs &a, int gq, cudaStream_t stream) {
  return a.geo.bits == 2 ? launch_b<2, false, false, true>(a, gq, stream) : launch_b<4, false, false, true>(a, gq, stream);
}

}  // namespace kvq
