// Instantiations of the batched union-of-active-rows kernel for __half weights.
#include "union_impl.cuh"

namespace sffn {
cudaError_t launch_union_f16(const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  return union_dispatch<__half>(cfg, a, grid, s);
}
}  // namespace sffn
