// Instantiations of the fused row-gather FFN kernel for __nv_bfloat16 rows.
#include "gather_impl.cuh"

namespace sffn {
cudaError_t launch_gather_bf16(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  return gather_dispatch<__nv_bfloat16>(cfg, a, grid, s);
}
}  // namespace sffn
