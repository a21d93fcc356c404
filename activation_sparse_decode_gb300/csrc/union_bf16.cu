// Instantiations of the batched union-of-active-rows kernel for __nv_bfloat16 weights.
#include "union_impl.cuh"

namespace sffn {
cudaError_t launch_union_bf16(const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  return union_dispatch<__nv_bfloat16>(cfg, a, grid, s);
}
}  // namespace sffn
