// Instantiations of the tensor-core batch kernels (union-of-active-rows FFN,
// predictor scores) for __half weights.
#include "score_mma.cuh"
#include "union_impl.cuh"

namespace sffn {
cudaError_t launch_union_f16(const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  return union_dispatch<__half>(cfg, a, grid, s);
}
cudaError_t launch_score_mma_f16(const ScoreMmaArgs& a, int bt, int grid, size_t smem, cudaStream_t s) {
  return score_mma_dispatch<__half>(a, bt, grid, smem, s);
}
}  // namespace sffn
