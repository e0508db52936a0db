// Split-kernel instantiations of the dithered INT8 scheme.
#include "decode_split.cuh"

namespace witcert {

cudaError_t decode_split_int8(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  return dispatch_flags<kInt8>(a, grid, st, pdl, occ);
}

}  // namespace witcert
