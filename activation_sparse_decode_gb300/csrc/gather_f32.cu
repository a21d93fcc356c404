// Instantiations of the fused row-gather FFN kernel for float rows.
#include "gather_impl.cuh"

namespace sffn {
cudaError_t launch_gather_f32(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  return gather_dispatch<float>(cfg, a, grid, s);
}
}  // namespace sffn
