// Instantiations of the single-launch decode layer kernel for __half weights.
#include "layer_impl.cuh"

namespace sffn {
cudaError_t launch_layer_f16(const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  return layer_dispatch<__half>(cfg, a, grid, s);
}
int layer_blocks_per_sm_f16(const LayerConfig& cfg) { return layer_blocks_per_sm_t<__half>(cfg); }
int layer_max_clusters_f16(const LayerConfig& cfg, int grid, int cs) { return layer_max_clusters_t<__half>(cfg, grid, cs); }
}  // namespace sffn
