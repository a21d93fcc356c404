// Small kernels around the sparse FFN: residual + LayerNorm between stacked
// layers, row permutation for the hot-first neuron order, the bounded-wait
// test hook, and the launch configuration of the gather kernel.

#include <algorithm>

#include "kernels.cuh"

namespace sffn {

cudaError_t launch_gather_f32(const GatherConfig&, const GatherArgs&, int, cudaStream_t);
cudaError_t launch_gather_f16(const GatherConfig&, const GatherArgs&, int, cudaStream_t);
cudaError_t launch_gather_bf16(const GatherConfig&, const GatherArgs&, int, cudaStream_t);

namespace {

constexpr int kLnThreads = 256;

__device__ float block_sum(float v, float* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_warp[w];  // fixed order
  return t;
}

// One block per token.  v = x + y in fp32; mean and biased variance by two
// passes; out = (v - mean) / sqrt(var + eps) * gamma + beta, rounded to T.
template <typename T>
__global__ void __launch_bounds__(kLnThreads)
    k_residual_ln(const T* __restrict__ x, const float* __restrict__ y, int d, const float* __restrict__ gamma,
                  const float* __restrict__ beta, float eps, T* out) {
  constexpr int E = Chunk<T>::N;
  __shared__ float s_warp[kLnThreads / 32];
  const T* xb = x + (size_t)blockIdx.x * d;
  const float* yb = y + (size_t)blockIdx.x * d;
  T* ob = out + (size_t)blockIdx.x * d;
  const int nch = d / E;
  auto load = [&](int ch, float* v) {
    unpack<T>(*reinterpret_cast<const uint4*>(xb + ch * E), v);
    const float4* yp = reinterpret_cast<const float4*>(yb + ch * E);
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 q = yp[e / 4];
      v[e] += q.x; v[e + 1] += q.y; v[e + 2] += q.z; v[e + 3] += q.w;
    }
  };
  float s = 0.f;
  for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
    float v[E];
    load(ch, v);
#pragma unroll
    for (int e = 0; e < E; ++e) s += v[e];
  }
  const float mean = block_sum(s, s_warp) / (float)d;
  float q = 0.f;
  for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
    float v[E];
    load(ch, v);
#pragma unroll
    for (int e = 0; e < E; ++e) q = fmaf(v[e] - mean, v[e] - mean, q);
  }
  const float var = block_sum(q, s_warp) / (float)d;
  const float rstd = 1.0f / sqrtf(var + eps);
  __syncthreads();  // every thread has read x before any (possibly in-place) write
  for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
    float v[E];
    load(ch, v);
    T o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float r = (v[e] - mean) * rstd;
      if (gamma != nullptr) r *= gamma[ch * E + e];
      if (beta != nullptr) r += beta[ch * E + e];
      o[e] = from_float<T>(r);
    }
    *reinterpret_cast<uint4*>(ob + ch * E) = *reinterpret_cast<const uint4*>(o);
  }
}

template <typename V>
__global__ void k_permute_rows(const V* __restrict__ src, V* __restrict__ dst, const int32_t* __restrict__ perm,
                               int rows, int64_t row_vec) {
  for (int i = blockIdx.x; i < rows; i += gridDim.x) {
    const int32_t from = perm[i];
    if (from < 0 || from >= rows) continue;  // not a permutation entry: leave the row alone
    const V* s = src + (int64_t)from * row_vec;
    V* o = dst + (int64_t)i * row_vec;
    for (int64_t k = threadIdx.x; k < row_vec; k += blockDim.x) o[k] = s[k];
  }
}

// Waits at the grid barrier for one more block than the grid has: the arrival
// never comes, so the wait must end by its limit with kStTimeout recorded.
__global__ void k_wait_timeout(WsHeader* hdr, uint32_t* flags, uint64_t limit_ns) {
  grid_barrier(hdr, flags, gridDim.x + 1u, barrier_generation(flags), limit_ns, 0x900u);
}

// Test hook: every block holds its SM's resources (its dynamic shared
// memory) for `ns` nanoseconds of wall time, then exits.  Bounded; touches
// no memory.
__global__ void k_occupy(uint64_t ns) {
  extern __shared__ unsigned char hold[];
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) __nanosleep(2000);
    hold[0] = 0;
  }
  __syncthreads();
}

template <typename T>
cudaError_t ln_launch(const void* x, const float* y, int B, int d, const float* gamma, const float* beta,
                      float eps, void* out, cudaStream_t s) {
  k_residual_ln<T><<<B, kLnThreads, 0, s>>>(static_cast<const T*>(x), y, d, gamma, beta, eps,
                                            static_cast<T*>(out));
  return cudaGetLastError();
}

int round_cpt(int cpt) {
  if (cpt <= 4) return std::max(cpt, 1);
  if (cpt <= 6) return 6;
  return 0;
}

}  // namespace

cudaError_t launch_residual_layernorm(int dtype, const void* x, const float* y, int B, int d,
                                      const float* gamma, const float* beta, float eps, void* x_out,
                                      cudaStream_t s) {
  switch (dtype) {
    case kF32: return ln_launch<float>(x, y, B, d, gamma, beta, eps, x_out, s);
    case kF16: return ln_launch<__half>(x, y, B, d, gamma, beta, eps, x_out, s);
    case kBF16: return ln_launch<__nv_bfloat16>(x, y, B, d, gamma, beta, eps, x_out, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_permute_rows(const void* src, void* dst, const int32_t* perm, int rows, int64_t row_bytes,
                                cudaStream_t s) {
  const int grid = std::min(rows, 65535);
  const bool vec16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  if (vec16)
    k_permute_rows<uint4><<<grid, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), perm, rows,
                                               row_bytes / 16);
  else
    k_permute_rows<uint32_t><<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst),
                                                  perm, rows, row_bytes / 4);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(WsHeader* hdr, uint32_t* flags, uint64_t limit_ns, cudaStream_t s) {
  k_wait_timeout<<<1, 32, 0, s>>>(hdr, flags, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_occupy(uint64_t ns, int blocks, size_t smem, cudaStream_t s) {
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_occupy, smem, &cur);
  if (e != cudaSuccess) return e;
  k_occupy<<<blocks, 32, smem, s>>>(ns);
  return cudaGetLastError();
}

int gather_max_bt(int dtype, int d) {
  const int E = dtype == kF32 ? 4 : 8;
  const int cpt = round_cpt((d / E + 255) / 256);
  if (cpt == 0) return 0;
  for (int bt : {4, 2, 1})
    if (bt * cpt * E <= 64) return bt;
  return 0;
}

bool gather_config(int dtype, int act, int d, int f, int bt, int grid, size_t smem_optin, GatherConfig* cfg) {
  const int esize = dtype == kF32 ? 4 : 2;
  const int E = 16 / esize;
  const int cpt = round_cpt((d / E + 255) / 256);
  if (cpt == 0 || bt * cpt * E > 64) return false;
  const size_t row_bytes = (size_t)d * esize;
  const size_t stage = (act == kReglu ? 3 : 2) * row_bytes;
  const int list_cap = (f + grid - 1) / grid + 1;
  const size_t list_bytes = ((size_t)list_cap * 9 + 15) / 16 * 16;  // neuron ids, biases, token bits
  const size_t static_smem = 8 * 1024;  // reduction scratch and scan words
  if (smem_optin < static_smem + list_bytes) return false;
  const size_t budget = smem_optin - static_smem - list_bytes;
  const size_t s = std::min<size_t>(16, budget / (stage + 8));
  if (s < 2) return false;
  cfg->threads = 256;
  cfg->cpt = cpt;
  cfg->bt = bt;
  cfg->nstages = (int)s;
  cfg->list_cap = list_cap;
  cfg->smem = s * stage + s * 8 + list_bytes;
  return true;
}

bool layer_config(int dtype, int act, int d, int f, int r, int grid, size_t smem_optin, bool balance,
                  LayerConfig* cfg) {
  const int esize = dtype == kF32 ? 4 : 2;
  const int E = 16 / esize;
  const int cpt = round_cpt((d / E + 255) / 256);
  if (cpt == 0 || cpt * E > 48) return false;  // x and y accumulators live in registers
  if (r / E > 4 * 32) return false;            // at most 4 chunks of a U row per lane
  const int own_cap = (f + grid - 1) / grid;
  const int nwords = (own_cap + 31) / 32;
  if (nwords > 256 || grid > 1024) return false;
  if (r > 32 * 32) return false;  // h slots: at most 32 per lane of the polling warp
  const size_t stage = (size_t)(act == kReglu ? 3 : 2) * d * esize;
  // h, stage barriers, own biases (2), list + list biases, words, activity
  // flags, the pair-exchange inbox, and the balancing scratch (3 x grid) when
  // the launches balance (the token stays in registers)
  const size_t bal = balance ? (size_t)grid * 12 : 0;
  const size_t inbox = (size_t)((own_cap + 1) & ~1) * 8 + 16;  // pair exchange entries, 16-byte aligned
  const size_t fixed = (size_t)((r + 3) & ~3) * 4 + 17 * 8 + (size_t)own_cap * 16 + nwords * 4 +
                       bal + (size_t)(own_cap + 15) / 16 * 16 + inbox + 80;
  const size_t reserve = 2048;  // static shared memory of the kernel
  if (smem_optin < fixed + reserve + 2 * stage) return false;
  const size_t budget = (smem_optin - fixed - reserve) / 16 * 16;
  const size_t s = std::min<size_t>(16, budget / stage);
  const size_t u_bytes = (size_t)own_cap * r * esize;
  cfg->cpt = cpt;
  cfg->act = act;
  cfg->nstages = (int)s;
  cfg->u_smem = u_bytes <= budget ? 1 : 0;
  cfg->region_bytes = (std::max(s * stage, cfg->u_smem ? u_bytes : 0) + 15) / 16 * 16;
  const size_t u_round = (u_bytes + 15) / 16 * 16;
  cfg->u_off = cfg->u_smem ? cfg->region_bytes - u_round : 0;  // U rows sit at the end of the region
  cfg->hot_stages = (int)std::min<size_t>(4, cfg->u_smem ? cfg->u_off / stage : s);
  cfg->balance = balance ? 1 : 0;
  cfg->smem = cfg->region_bytes + (size_t)((r + 3) & ~3) * 4 + (s + 1) * 8 +
              (size_t)own_cap * 16 + nwords * 4 + (size_t)(own_cap + 15) / 16 * 16 + inbox + bal + 80;
  return cfg->smem + reserve <= smem_optin;
}

bool union_config(int dtype, int act, int d, int f, int B, int grid, size_t smem_optin, UnionConfig* cfg) {
  if (dtype != kF16 && dtype != kBF16) return false;  // 16-bit tensor-core operands
  if (d % 128 != 0 || B < 1 || B > 32) return false;
  const int W = (f + 31) / 32;
  if (W > kUnionMaxWpt * kUnionThreads) return false;
  const int bt = B <= 8 ? 8 : B <= 16 ? 16 : 32;
  const int n1 = std::max(16, bt);
  const int nm = act == kReglu ? 2 : 1;
  const int list_cap = (f + grid - 1) / grid + 1;
  if ((size_t)(list_cap + 1) * 8 > kUnionAtBytes) return false;  // word list scratch
  const size_t max_slot = std::max<size_t>(((size_t)nm * 128 + n1) * 128, 128 * 256);
  const size_t lists = ((size_t)list_cap * 12 + 1023) / 1024 * 1024;  // neuron, token bits, bias
  const size_t reserve = 2048;                                        // static shared memory
  if (smem_optin < reserve + kUnionAtBytes + lists + 2 * max_slot) return false;
  const size_t ring = std::min<size_t>(kUnionMaxSlots * max_slot,
                                       (smem_optin - reserve - kUnionAtBytes - lists) / 1024 * 1024);
  cfg->bt = bt;
  cfg->list_cap = list_cap;
  cfg->ring_bytes = ring;
  cfg->smem = ring + kUnionAtBytes + lists;
  return true;
}

cudaError_t launch_union_f16(const UnionConfig&, const UnionArgs&, int, cudaStream_t);
cudaError_t launch_union_bf16(const UnionConfig&, const UnionArgs&, int, cudaStream_t);

cudaError_t launch_union(int dtype, const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  switch (dtype) {
    case kF16: return launch_union_f16(cfg, a, grid, s);
    case kBF16: return launch_union_bf16(cfg, a, grid, s);
  }
  return cudaErrorInvalidValue;
}

bool score_mma_config(int dtype, int r, int B, size_t smem_optin, size_t* ring_bytes) {
  if (dtype != kF16 && dtype != kBF16) return false;
  if (r % 64 != 0 || B < 1 || B > 32) return false;
  const int bt = B <= 8 ? 8 : B <= 16 ? 16 : 32;
  const size_t slot = 128 * 128 + (size_t)((3 * bt + 15) / 16 * 16) * 128;
  const size_t reserve = 2048;  // static shared memory
  if (smem_optin < reserve + 2 * slot) return false;
  *ring_bytes = std::min<size_t>(32 * slot, (smem_optin - reserve) / slot * slot);
  return true;
}

cudaError_t launch_score_mma_f16(const ScoreMmaArgs&, int, int, size_t, cudaStream_t);
cudaError_t launch_score_mma_bf16(const ScoreMmaArgs&, int, int, size_t, cudaStream_t);

cudaError_t launch_score_mma(int dtype, const ScoreMmaArgs& a, int bt, int grid, cudaStream_t s) {
  switch (dtype) {
    case kF16: return launch_score_mma_f16(a, bt, grid, a.ring_bytes, s);
    case kBF16: return launch_score_mma_bf16(a, bt, grid, a.ring_bytes, s);
  }
  return cudaErrorInvalidValue;
}

int layer_blocks_per_sm_f32(const LayerConfig&);
int layer_blocks_per_sm_f16(const LayerConfig&);
int layer_blocks_per_sm_bf16(const LayerConfig&);

int layer_max_clusters_f32(const LayerConfig&, int, int);
int layer_max_clusters_f16(const LayerConfig&, int, int);
int layer_max_clusters_bf16(const LayerConfig&, int, int);

int layer_max_clusters(int dtype, const LayerConfig& cfg, int grid, int cs) {
  switch (dtype) {
    case kF32: return layer_max_clusters_f32(cfg, grid, cs);
    case kF16: return layer_max_clusters_f16(cfg, grid, cs);
    case kBF16: return layer_max_clusters_bf16(cfg, grid, cs);
  }
  return 0;
}

int layer_blocks_per_sm(int dtype, const LayerConfig& cfg) {
  switch (dtype) {
    case kF32: return layer_blocks_per_sm_f32(cfg);
    case kF16: return layer_blocks_per_sm_f16(cfg);
    case kBF16: return layer_blocks_per_sm_bf16(cfg);
  }
  return 0;
}

cudaError_t launch_layer_f32(const LayerConfig&, const LayerArgs&, int, cudaStream_t);
cudaError_t launch_layer_f16(const LayerConfig&, const LayerArgs&, int, cudaStream_t);
cudaError_t launch_layer_bf16(const LayerConfig&, const LayerArgs&, int, cudaStream_t);

cudaError_t launch_layer(int dtype, const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  switch (dtype) {
    case kF32: return launch_layer_f32(cfg, a, grid, s);
    case kF16: return launch_layer_f16(cfg, a, grid, s);
    case kBF16: return launch_layer_bf16(cfg, a, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gather(int dtype, const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  switch (dtype) {
    case kF32: return launch_gather_f32(cfg, a, grid, s);
    case kF16: return launch_gather_f16(cfg, a, grid, s);
    case kBF16: return launch_gather_bf16(cfg, a, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sffn
