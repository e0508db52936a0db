// Split-kernel instantiations of KIVI-style 2-bit.
#include "decode_split.cuh"

namespace witcert {

cudaError_t decode_split_kivi(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  return dispatch_flags<kKivi>(a, grid, st, pdl, occ);
}

}  // namespace witcert
