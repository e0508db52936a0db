// Split-kernel instantiations of raw-cast FP8-E4M3.
#include "decode_split.cuh"

namespace witcert {

cudaError_t decode_split_fp8(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  return dispatch_flags<kFp8>(a, grid, st, pdl, occ);
}

}  // namespace witcert
