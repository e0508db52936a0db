// Split-kernel instantiations of INT8 round to nearest.
#include "decode_split.cuh"

namespace witcert {

cudaError_t decode_split_rtn(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  return dispatch_flags<kRtn>(a, grid, st, pdl, occ);
}

}  // namespace witcert
