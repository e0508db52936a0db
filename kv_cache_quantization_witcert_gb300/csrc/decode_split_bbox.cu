// Split-kernel instantiations of the black-box bf16 store.
#include "decode_split.cuh"

namespace witcert {

cudaError_t decode_split_bbox(const DecodeArgs& a, dim3 grid, cudaStream_t st, bool pdl, int* occ) {
  return dispatch_flags<kBbox>(a, grid, st, pdl, occ);
}

}  // namespace witcert
