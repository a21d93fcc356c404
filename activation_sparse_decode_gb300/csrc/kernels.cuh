// Launchers of the sparse-FFN kernels (host side, used by the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace sffn {

// ---- predictor hidden layer: h[b][k] = sum_j V[k][j] x[b][j]
struct PredHiddenArgs {
  const void* V;       // [r][d]
  const void* x;       // [B][d]
  int B, r, d;
  int kc_elems;        // elements of d per K-chunk (multiple of 32 chunks' worth)
  int KS;              // number of K-chunks
  float* h_part;       // [KS][B][r] partial sums (workspace)
  float* h;            // [B][r] final (workspace)
  uint32_t* tickets;   // [row groups][token groups] arrival counters (zeroed)
  void* h3;            // NULL, or [3*bt][r] dtype: h split into hi, mid, lo 16-bit parts (rows part*bt + b)
  int bt;              // 0: tokens per block chosen from B; else 8, 16 or 32 (one token group)
  int cluster = 0;     // 1: the cluster kernel (16-bit weights, h3 set, bt >= B, d a multiple of 512)
};
int pred_hidden_row_groups(int r);
// Dynamic shared memory of the cluster hidden-layer kernel (0: d does not fit its split).
size_t pred_hidden_cluster_smem(int d, int bt);
cudaError_t launch_pred_hidden(int dtype, const PredHiddenArgs& a, cudaStream_t s);

// ---- predictor scores + threshold: mask[b][w] bit j  <=>  U[32w+j].h[b] + pb > tau
struct PredScoreArgs {
  const void* U;       // [f][r]
  const float* h;      // [B][r]
  const float* pb;     // [f]
  float tau;
  int B, f, r, W;      // W = ceil(f / 32) mask words per token
  uint32_t* mask;      // [B][W]
  float* scores;       // NULL or [B][f]
  int grid;            // blocks (grid-stride over 64-row blocks)
};
cudaError_t launch_pred_score(int dtype, const PredScoreArgs& a, cudaStream_t s);

// ---- compaction: ascending active-index list per token
cudaError_t launch_compact(const uint32_t* mask, int B, int f, int W, int32_t* idx, int32_t* n_active,
                           cudaStream_t s);

// ---- counts[i] += number of tokens with bit i set
cudaError_t launch_count_bits(const uint32_t* mask, int B, int f, int W, int32_t* counts, cudaStream_t s);

// ---- fused row-gather FFN (CUDA cores, up to 4 tokens per pass)
struct GatherArgs {
  const void* x;        // [B][d] tokens of this pass
  const void* w_up;
  const void* w_gate;   // ReGLU only
  const void* w_downT;
  const float* b;       // NULL or [f]
  const uint32_t* mask; // [B][W] predicted bits of this pass (ignored when dense)
  float* y;             // [B][d]
  float* y_part;        // [grid][B][d] per-block partial outputs (workspace)
  WsHeader* hdr;
  uint32_t* bar_flags;  // [grid] grid-barrier release flags, 128 bytes apart (workspace)
  int B, d, f, W;
  int act;              // Act
  int dense;            // 1: every neuron (no predictor)
  int nstages;          // pipeline depth (>= 2)
  int list_cap;         // per-block capacity of the local neuron list
  uint64_t wait_ns;
  size_t wstride;       // bytes from one neuron's row to the next in each weight matrix
};
struct GatherConfig {
  int threads, cpt, bt, nstages, list_cap;
  size_t smem;
};
// Largest tokens-per-pass the register budget allows for this row width.
int gather_max_bt(int dtype, int d);
bool gather_config(int dtype, int act, int d, int f, int bt, int grid, size_t smem_optin,
                   GatherConfig* cfg);
cudaError_t launch_gather(int dtype, const GatherConfig& cfg, const GatherArgs& a, int grid,
                          cudaStream_t s);

// ---- one token through one layer in a single launch (predictor + gather)
struct LayerArgs {
  const void* x;          // [d] the token, or x_prev when y_prev is given
  const float* y_prev;    // NULL, or the previous layer's output: x := round(LN(x_prev + y_prev))
  void* x_ln_out;         // with y_prev: where the formed x is stored ([d], may be NULL)
  const float* ln_gamma;  // NULL = 1
  const float* ln_beta;   // NULL = 0
  float ln_eps;
  const void* V;          // [r][d]
  const void* U;          // [f][r]
  const float* pb;        // [f] predictor bias
  const float* b;         // NULL or [f] gated bias
  float tau;
  const void* w_up;
  const void* w_gate;
  const void* w_downT;
  float* y;               // [d] output, zeroed and accumulated here
  unsigned long long* h_slots;  // [r][16] {launch tag, h value} in word 0 of each 128-byte line (workspace)
  uint32_t* mask;         // NULL or [ceil(f/32)] words, zeroed and set here
  WsHeader* hdr;
  uint32_t* bar_flags;    // [grid] grid-barrier release flags, 128 bytes apart
  int d, f, r, act, nstages, u_smem;
  int hot_rows;           // neurons [0, hot_rows) are prefetched before the predictor decides
  int warm_rows;          // neurons [0, warm_rows): rows warmed in L2 while the predictor runs
  int hot_stages;         // ring stages free of the U rows, usable for that prefetch
  int balance;            // 1: even out the active rows over the blocks (second barrier)
  int cluster;            // > 1: launched in clusters of this many blocks, which even out their rows
  int static_weights;     // 1: the weights are read before the dependency wait (never written by kernels)
  int prefill;            // own rows each block starts streaming before the balancing
  uint64_t* bal_counts;   // [grid] {epoch, active rows} per block (workspace)
  int32_t* bal_lists;     // [grid][own_cap] {neuron, bias bits} pairs per block (workspace)
  size_t region_bytes;
  size_t u_off;           // offset of the staged U rows inside the region
  uint64_t wait_ns;
  // Look-ahead (stacks at batch 1): this call's active rows come from la_in,
  // predicted by the previous call, and the predictor fields above (V, U,
  // pb, tau) are the NEXT layer's, evaluated on this call's input into la_out.
  const uint32_t* la_in;  // NULL, or [ceil(f/32)] mask words of this call
  uint32_t* la_out;       // [ceil(f/32)] mask words for the next call (zeroed and set here)
  int predict_only;       // 1: only the predictor, into la_out: no rows read, no y (launched without clusters)
  size_t wstride;         // bytes from one neuron's row to the next in each weight matrix
};
struct LayerConfig {
  int cpt, act, nstages, u_smem, hot_stages;
  int balance;  // 1: shared memory holds the balancing scratch
  size_t region_bytes, u_off, smem;
};
bool layer_config(int dtype, int act, int d, int f, int r, int grid, size_t smem_optin, bool balance,
                  LayerConfig* cfg);
// Workspace bytes of the layer kernel's h slots: one {tag, h value} word per
// rank row, each on its own 128-byte line.
inline size_t layer_slot_bytes(int r) { return (size_t)r * 128; }
cudaError_t launch_layer(int dtype, const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s);
// Blocks of the layer kernel that can be resident on one SM with this configuration.
int layer_blocks_per_sm(int dtype, const LayerConfig& cfg);
// Clusters of cs blocks of the layer kernel that can be resident at once.
int layer_max_clusters(int dtype, const LayerConfig& cfg, int grid, int cs);

// ---- batched decode over the union of the tokens' active rows (tensor cores)
struct UnionArgs {
  const void* x;          // [B][d] tokens
  const void* w_up;
  const void* w_gate;     // ReGLU only
  const void* w_downT;
  const float* b;         // NULL or [f]
  const uint32_t* mask;   // [B][W] predicted bits
  float* y;               // [B][d]: zero on entry, accumulated with float atomics
  WsHeader* hdr;
  int B, d, f, W, act;
  int list_cap;           // >= the most union members one block can get
  size_t ring_bytes;      // shared memory of the copy ring
  uint64_t wait_ns;
  size_t wstride;         // bytes from one neuron's row to the next in each weight matrix
};
constexpr int kUnionThreads = 416;       // 4 epilogue warps, 1 MMA warp, 8 copy warps
constexpr int kUnionMaxWpt = 4;          // mask words per thread in the union scan
constexpr int kUnionMaxSlots = 32;
constexpr size_t kUnionAtBytes = 17408;  // GEMM2 B operand (128 neurons x 64 columns x 2 bytes, padded)
struct UnionConfig {
  int bt;                 // token columns of the tiles: 8, 16 or 32
  int list_cap;
  size_t ring_bytes, smem;
};
bool union_config(int dtype, int act, int d, int f, int B, int grid, size_t smem_optin, UnionConfig* cfg);
cudaError_t launch_union(int dtype, const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s);

// ---- batched predictor scores on the tensor cores (8 to 32 tokens)
struct ScoreMmaArgs {
  const void* U;        // [f][r] dtype
  const void* h3;       // [3*bt][r] dtype: the tokens' hidden vectors as hi, mid, lo parts
  const float* pb;      // [f]
  float tau;
  int B, f, r, W;
  uint32_t* mask;       // [B][W] out
  WsHeader* hdr;
  size_t ring_bytes;
  uint64_t wait_ns;
};
constexpr int kScoreMmaThreads = 416;
bool score_mma_config(int dtype, int r, int B, size_t smem_optin, size_t* ring_bytes);
cudaError_t launch_score_mma(int dtype, const ScoreMmaArgs& a, int bt, int grid, cudaStream_t s);

// ---- residual + LayerNorm: x_out = round(LN(x + y) * gamma + beta)
cudaError_t launch_residual_layernorm(int dtype, const void* x, const float* y, int B, int d,
                                      const float* gamma, const float* beta, float eps, void* x_out,
                                      cudaStream_t s);

// ---- dst[i] = src[perm[i]] rows
cudaError_t launch_permute_rows(const void* src, void* dst, const int32_t* perm, int rows,
                                int64_t row_bytes, cudaStream_t s);

// ---- test hook: a barrier wait that cannot complete
cudaError_t launch_wait_timeout(WsHeader* hdr, uint32_t* flags, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_occupy(uint64_t ns, int blocks, size_t smem, cudaStream_t s);

// ---- dense fallback (every row, two library GEMMs): the masked activation
// between them (16-bit high part and remainder, [2B][f]) and the sum of the
// two halves of the second product into y
cudaError_t launch_dense_act(int dtype, const float* d_up, const float* d_gate, const float* bias,
                             const uint32_t* mask, int B, int f, int W, void* A, cudaStream_t s);
cudaError_t launch_dense_combine(const float* y2, int B, int d, float* y, cudaStream_t s);

}  // namespace sffn
