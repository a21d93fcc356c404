// One decode token through one FFN layer in a single launch: predictor,
// threshold, neuron-aware row gather, activation and down projection.
//
// Why one kernel.  At batch 1 a layer moves only tens of MB, a few microseconds
// of HBM time, so the cost of separate launches and of their dependency gaps is
// as large as the work.  Here every block works through all phases and the
// only grid-wide synchronisation is a single bounded barrier between the
// predictor's hidden layer (h = V x, split over all blocks) and its scores.
//
// Neuron ownership.  Block c of G owns the neurons i = c, c + G, c + 2G, ...
// It scores exactly its own neurons (their rows of U), so it learns its own
// active set without any mask exchange, and gathers only its own active rows.
// With the hot-first order the always-active neurons are spread round-robin
// over the blocks, so each block expects the same number of active rows
// (PowerInfer's offline hot/cold placement, here placing neurons on SMs
// instead of on GPU vs CPU: PowerInfer page, "Politica de colocacion de
// neuronas").
//
// Overlap.  At t = 0 each block issues bulk copies of its U rows into shared
// memory, an L2 prefetch of the V tiles it will stream, and loads of its
// biases, so the predictor's 2-3 weight streams are in flight together.  The
// rows of active neurons follow the same cp.async.bulk + mbarrier ring as the
// gather kernel.  The down projection's per-block partial output is added into
// y with vector float atomics (y is zeroed in the first phase, before the
// barrier), so there is no second grid-wide step.
//
// Stacked layers: when y_prev is given, the block first forms this layer's
// input x = round(LayerNorm(x_prev + y_prev)) itself (every block computes the
// same values; each writes its slice of the stored result), so no separate
// LayerNorm launch sits between layers.
#pragma once

#include "kernels.cuh"

namespace sffn {

constexpr int kLayerThreads = 256;
constexpr int kLayerWarps = kLayerThreads / 32;

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ float layer_block_sum(float v, float* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kLayerWarps; ++w) t += s_warp[w];
  return t;
}

template <typename T>
__device__ __forceinline__ void pack_store(T* dst, const float* v);
template <>
__device__ __forceinline__ void pack_store<float>(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void pack_store<__half>(__half* dst, const float* v) {
  __half o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = __float2half_rn(v[e]);
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
}
template <>
__device__ __forceinline__ void pack_store<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  __nv_bfloat16 o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = __float2bfloat16_rn(v[e]);
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
}

template <typename T, int CPT>
__global__ void __launch_bounds__(kLayerThreads, 1) k_layer(const LayerArgs a) {
  constexpr int CPL = 4;  // up to 4 16-byte chunks of a U row per lane (rank <= 128 * elements per chunk)
  constexpr int E = Chunk<T>::N;
  constexpr int ES = sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_red[2][kLayerWarps][2];
  __shared__ float s_warp[kLayerWarps];
  __shared__ int s_nloc;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int d = a.d, f = a.f, r = a.r;
  const int NCH = d / E;       // 16-byte chunks per d-row
  const int NC = r / E;        // 16-byte chunks per U row
  const uint32_t row_bytes = (uint32_t)d * ES;
  const uint32_t urow_bytes = (uint32_t)r * ES;
  const bool reglu = a.act == kReglu;
  const int nrows = reglu ? 3 : 2;
  const uint32_t stage_bytes = nrows * row_bytes;
  const int S = a.nstages;
  const int n_own = c < f ? (f - c + G - 1) / G : 0;
  const int own_cap = (f + G - 1) / G;
  const int nwords = (own_cap + 31) / 32;

  // ---- shared memory carve-up (offsets are multiples of 16)
  unsigned char* region = smem;  // U rows (phases 0-4), then the row ring
  T* xs = reinterpret_cast<T*>(smem + a.region_bytes);
  float* hs = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(xs) + (size_t)d * ES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(hs + ((r + 3) & ~3));
  float* ownb = reinterpret_cast<float*>(bars + S + 1);
  float* ownpb = ownb + own_cap;
  uint32_t* words = reinterpret_cast<uint32_t*>(ownpb + own_cap);
  int32_t* list = reinterpret_cast<int32_t*>(words + nwords);
  uint64_t* ubar = bars + S;

  // ---- phase 0: start every independent stream, zero the outputs
  if (tid == 0) {
    for (int s = 0; s <= S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (a.u_smem && n_own > 0) {
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(ubar, (uint32_t)n_own * urow_bytes);
      const unsigned char* U = static_cast<const unsigned char*>(a.U);
      for (int j = 0; j < n_own; ++j)
        bulk_g2s(region + (size_t)j * urow_bytes, U + (size_t)(c + (size_t)j * G) * urow_bytes, urow_bytes, ubar, pol);
    }
  }
  {  // L2 prefetch of this block's V tiles (one row segment per thread)
    const int tiles = a.RG * a.KS;
    const unsigned char* V = static_cast<const unsigned char*>(a.V);
    for (int tile = c; tile < tiles; tile += G) {
      const int rg = tile / a.KS, ks = tile - rg * a.KS;
      const int k0 = ks * a.kc, kn = min(a.kc, d - k0);
      const int row = rg * 16 + tid;
      if (tid < 16 && row < r) bulk_prefetch_l2(V + ((size_t)row * d + k0) * ES, (uint32_t)kn * ES);
    }
  }
  for (int j = tid; j < n_own; j += kLayerThreads) {
    const int i = c + j * G;
    ownb[j] = a.b != nullptr ? __ldg(&a.b[i]) : 0.f;
    ownpb[j] = __ldg(&a.pb[i]);
  }
  {
    float4* y4 = reinterpret_cast<float4*>(a.y);
    const int N4 = d / 4;
    for (int q = (int)((int64_t)N4 * c / G) + tid; q < (int)((int64_t)N4 * (c + 1) / G); q += kLayerThreads)
      y4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.mask != nullptr) {
      const int W = (f + 31) / 32;
      for (int w = (int)((int64_t)W * c / G) + tid; w < (int)((int64_t)W * (c + 1) / G); w += kLayerThreads)
        a.mask[w] = 0u;
    }
  }
  // the token: loaded, or formed from the previous layer by residual + LayerNorm
  if (a.y_prev == nullptr) {
    const uint4* xg = static_cast<const uint4*>(a.x);
    for (int ch = tid; ch < NCH; ch += kLayerThreads) reinterpret_cast<uint4*>(xs)[ch] = xg[ch];
  } else {
    const T* xp = static_cast<const T*>(a.x);
    auto load = [&](int ch, float* v) {
      unpack<T>(*reinterpret_cast<const uint4*>(xp + ch * E), v);
      const float4* yp = reinterpret_cast<const float4*>(a.y_prev + ch * E);
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 q = __ldcg(&yp[e / 4]);
        v[e] += q.x; v[e + 1] += q.y; v[e + 2] += q.z; v[e + 3] += q.w;
      }
    };
    float s = 0.f;
    for (int ch = tid; ch < NCH; ch += kLayerThreads) {
      float v[E];
      load(ch, v);
#pragma unroll
      for (int e = 0; e < E; ++e) s += v[e];
    }
    const float mean = layer_block_sum(s, s_warp) / (float)d;
    float q = 0.f;
    for (int ch = tid; ch < NCH; ch += kLayerThreads) {
      float v[E];
      load(ch, v);
#pragma unroll
      for (int e = 0; e < E; ++e) q = fmaf(v[e] - mean, v[e] - mean, q);
    }
    const float var = layer_block_sum(q, s_warp) / (float)d;
    const float rstd = 1.0f / sqrtf(var + a.ln_eps);
    for (int ch = tid; ch < NCH; ch += kLayerThreads) {
      float v[E];
      load(ch, v);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        float o = (v[e] - mean) * rstd;
        if (a.ln_gamma != nullptr) o *= a.ln_gamma[ch * E + e];
        if (a.ln_beta != nullptr) o += a.ln_beta[ch * E + e];
        v[e] = o;
      }
      pack_store<T>(xs + ch * E, v);
    }
  }
  __syncthreads();
  if (a.y_prev != nullptr && a.x_ln_out != nullptr) {  // each block stores its slice of the new x
    uint4* xo = static_cast<uint4*>(a.x_ln_out);
    for (int ch = (int)((int64_t)NCH * c / G) + tid; ch < (int)((int64_t)NCH * (c + 1) / G); ch += kLayerThreads)
      xo[ch] = reinterpret_cast<const uint4*>(xs)[ch];
  }

  // ---- phase 1: partial h over this block's (16-row, K-chunk) tiles of V
  {
    const T* V = static_cast<const T*>(a.V);
    const int tiles = a.RG * a.KS;
    for (int tile = c; tile < tiles; tile += G) {
      const int rg = tile / a.KS, ks = tile - rg * a.KS;
      const int k0 = ks * a.kc;
      const int nch = min(a.kc, d - k0) / E;
      const int row0 = rg * 16 + warp * 2;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
      for (int ch = lane; ch < nch; ch += 32) {
        const uint4 r0 = row0 < r ? ldg_stream(V + (size_t)row0 * d + k0 + ch * E) : make_uint4(0, 0, 0, 0);
        const uint4 r1 = row0 + 1 < r ? ldg_stream(V + (size_t)(row0 + 1) * d + k0 + ch * E) : make_uint4(0, 0, 0, 0);
        float xv[E], w0[E], w1[E];
        unpack<T>(reinterpret_cast<const uint4*>(xs + k0)[ch], xv);
        unpack<T>(r0, w0);
        unpack<T>(r1, w1);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          acc0 = fmaf(w0[e], xv[e], acc0);
          acc1 = fmaf(w1[e], xv[e], acc1);
        }
      }
      acc0 = warp_sum(acc0);
      acc1 = warp_sum(acc1);
      if (lane == 0) {
        if (row0 < r) a.h_part[(size_t)ks * r + row0] = acc0;
        if (row0 + 1 < r) a.h_part[(size_t)ks * r + row0 + 1] = acc1;
      }
    }
  }

  // ---- phase 2: every block's partials are in place
  if (!grid_barrier(a.hdr, (uint32_t)G, a.wait_ns, 0x300u)) {
    if (tid == 0 && a.u_smem && n_own > 0) mbar_wait(ubar, 0, a.hdr, a.wait_ns, 0x301u);
    return;
  }

  // ---- phase 3: h = sum of the K-chunk partials (fixed order)
  for (int k = tid; k < r; k += kLayerThreads) {
    float s = 0.f;
    for (int ks = 0; ks < a.KS; ++ks) s += __ldcg(&a.h_part[(size_t)ks * r + k]);
    hs[k] = s;
  }
  __syncthreads();

  // ---- phase 4: scores of the owned neurons, 32 rows per warp task; lane k
  // ends up with row k's full dot product (reduce-scatter over the lanes)
  bool u_ok = true;
  if (a.u_smem && n_own > 0) u_ok = mbar_wait(ubar, 0, a.hdr, a.wait_ns, 0x302u);
  if (__syncthreads_or(!u_ok)) return;
  {
    float hreg[CPL][E];
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
      const int ch = lane + 32 * cc;
#pragma unroll
      for (int e = 0; e < E; ++e) hreg[cc][e] = ch < NC ? hs[ch * E + e] : 0.f;
    }
    const T* Ug = static_cast<const T*>(a.U);
    for (int q = warp; q < nwords; q += kLayerWarps) {
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = q * 32 + k;
        float acc = 0.f;
        if (j < n_own) {
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) {
            const int ch = lane + 32 * cc;
            if (ch < NC) {
              const uint4 raw = a.u_smem ? reinterpret_cast<const uint4*>(region + (size_t)j * urow_bytes)[ch]
                                         : ldg_stream(Ug + (size_t)(c + (size_t)j * G) * r + ch * E);
              float w[E];
              unpack<T>(raw, w);
#pragma unroll
              for (int e = 0; e < E; ++e) acc = fmaf(w[e], hreg[cc][e], acc);
            }
          }
        }
        v[k] = acc;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < o; ++k) {
          const float send = upper ? v[k] : v[k + o];
          const float keep = upper ? v[k + o] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const int j = q * 32 + lane;
      const bool act = j < n_own && (v[0] + ownpb[j < n_own ? j : 0]) > a.tau;
      const uint32_t bits = __ballot_sync(0xffffffffu, act);
      if (lane == 0) words[q] = bits;
      if (act && a.mask != nullptr) {
        const int i = c + j * G;
        atomicOr(&a.mask[i >> 5], 1u << (i & 31));
      }
    }
  }
  __syncthreads();
  // ascending list of active owned rows
  if (tid < nwords) {
    int pre = 0;
    for (int w = 0; w < tid; ++w) pre += __popc(words[w]);
    uint32_t bits = words[tid];
    while (bits) {
      const int k = __ffs(bits) - 1;
      bits &= bits - 1;
      list[pre++] = tid * 32 + k;
    }
    if (tid == nwords - 1) s_nloc = pre;
  }
  if (nwords == 0 && tid == 0) s_nloc = 0;
  __syncthreads();
  const int nloc = s_nloc;

  // ---- phase 5: stream the active rows through the ring, accumulate
  const unsigned char* gup = static_cast<const unsigned char*>(a.w_up);
  const unsigned char* ggt = static_cast<const unsigned char*>(a.w_gate);
  const unsigned char* gdn = static_cast<const unsigned char*>(a.w_downT);
  uint64_t policy = 0;
  if (tid == 0) policy = policy_evict_first();
  auto issue = [&](int j) {
    const int s = j % S;
    const size_t off = (size_t)(c + (size_t)list[j] * G) * row_bytes;
    unsigned char* dst = region + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&bars[s], stage_bytes);
    bulk_g2s(dst, gup + off, row_bytes, &bars[s], policy);
    if (reglu) bulk_g2s(dst + row_bytes, ggt + off, row_bytes, &bars[s], policy);
    bulk_g2s(dst + (size_t)(nrows - 1) * row_bytes, gdn + off, row_bytes, &bars[s], policy);
  };
  if (tid == 0)
    for (int j = 0; j < min(S, nloc); ++j) issue(j);

  float xr[CPT][E], yacc[CPT][E];
#pragma unroll
  for (int cq = 0; cq < CPT; ++cq) {
    const int ch = tid + cq * kLayerThreads;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (ch < NCH) raw = reinterpret_cast<const uint4*>(xs)[ch];
    unpack<T>(raw, xr[cq]);
#pragma unroll
    for (int e = 0; e < E; ++e) yacc[cq][e] = 0.f;
  }
  int consumed = 0;
  bool failed = false;
  for (int j = 0; j < nloc; ++j) {
    const int s = j % S;
    const bool ok = mbar_wait(&bars[s], (uint32_t)(j / S) & 1u, a.hdr, a.wait_ns, 0x303u);
    const uint4* up = reinterpret_cast<const uint4*>(region + (size_t)s * stage_bytes);
    const uint4* gt = up + NCH;
    const uint4* dn = up + (size_t)(nrows - 1) * NCH;
    float pu = 0.f, pg = 0.f;
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      if (ch < NCH) {
        float w[E];
        unpack<T>(up[ch], w);
#pragma unroll
        for (int e = 0; e < E; ++e) pu = fmaf(w[e], xr[cq][e], pu);
        if (reglu) {
          unpack<T>(gt[ch], w);
#pragma unroll
          for (int e = 0; e < E; ++e) pg = fmaf(w[e], xr[cq][e], pg);
        }
      }
    }
    pu = warp_sum(pu);
    if (reglu) pg = warp_sum(pg);
    if (lane == 0) {
      s_red[j & 1][warp][0] = pu;
      s_red[j & 1][warp][1] = pg;
    }
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    consumed = j + 1;
    if (tid == 0 && j >= 1 && j - 1 + S < nloc) issue(j - 1 + S);
    float u = 0.f, g = 0.f;
#pragma unroll
    for (int w = 0; w < kLayerWarps; ++w) {
      u += s_red[j & 1][w][0];
      g += s_red[j & 1][w][1];
    }
    const float bias = ownb[list[j]];
    const float act = reglu ? fmaxf(g + bias, 0.f) * u : fmaxf(u + bias, 0.f);
    if (act != 0.f) {
#pragma unroll
      for (int cq = 0; cq < CPT; ++cq) {
        const int ch = tid + cq * kLayerThreads;
        if (ch < NCH) {
          float w[E];
          unpack<T>(dn[ch], w);
#pragma unroll
          for (int e = 0; e < E; ++e) yacc[cq][e] = fmaf(act, w[e], yacc[cq][e]);
        }
      }
    }
  }
  if (failed) {
    if (tid == 0) {
      const int issued = consumed == 0 ? min(S, nloc) : min(nloc, consumed - 1 + S);
      for (int j = consumed; j < issued; ++j)
        mbar_wait(&bars[j % S], (uint32_t)(j / S) & 1u, a.hdr, a.wait_ns, 0x304u);
    }
    return;
  }

  // ---- phase 6: add this block's contribution into y
  if (nloc > 0) {
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      if (ch < NCH) {
        float4* o = reinterpret_cast<float4*>(a.y + (size_t)ch * E);
#pragma unroll
        for (int e = 0; e < E; e += 4)
          atomicAdd(&o[e / 4], make_float4(yacc[cq][e], yacc[cq][e + 1], yacc[cq][e + 2], yacc[cq][e + 3]));
      }
    }
  }
}

template <typename T, int CPT>
cudaError_t layer_launch(const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_layer<T, CPT>, cfg.smem, &cur);
  if (e != cudaSuccess) return e;
  k_layer<T, CPT><<<grid, kLayerThreads, cfg.smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t layer_dispatch(const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  switch (cfg.cpt) {
    case 1: return layer_launch<T, 1>(cfg, a, grid, s);
    case 2: return layer_launch<T, 2>(cfg, a, grid, s);
    case 3: return layer_launch<T, 3>(cfg, a, grid, s);
    case 4: return layer_launch<T, 4>(cfg, a, grid, s);
    case 6: return layer_launch<T, 6>(cfg, a, grid, s);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace sffn
