// Instantiations of the single-launch decode layer kernel for __nv_bfloat16 weights.
#include "layer_impl.cuh"

namespace sffn {
cudaError_t launch_layer_bf16(const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  return layer_dispatch<__nv_bfloat16>(cfg, a, grid, s);
}
int layer_blocks_per_sm_bf16(const LayerConfig& cfg) { return layer_blocks_per_sm_t<__nv_bfloat16>(cfg); }
int layer_max_clusters_bf16(const LayerConfig& cfg, int grid, int cs) { return layer_max_clusters_t<__nv_bfloat16>(cfg, grid, cs); }
}  // namespace sffn
