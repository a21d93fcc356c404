// Instantiations of the fused row-gather FFN kernel for __half rows.
#include "gather_impl.cuh"

namespace sffn {
cudaError_t launch_gather_f16(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  return gather_dispatch<__half>(cfg, a, grid, s);
}
}  // namespace sffn
