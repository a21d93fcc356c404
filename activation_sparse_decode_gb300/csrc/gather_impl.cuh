// Fused row-gather FFN for decode: for every neuron predicted active, read its
// row of W_up (and W_gate) and its row of W_down^T once, compute the activation
// and accumulate a_i * W_down^T[i, :] -- the neuron-aware operator that works on
// single row vectors of a matrix (PowerInfer page, "Operador consciente de
// neuronas"), built so that skipped rows are never read (sparsity page, the
// opening section: rows whose ReLU output is zero contribute nothing, and
// skipping them saves DRAM-to-cache traffic).
//
// GB300 design.  One block per SM, persistent over its share of the active
// list.  Every block rebuilds the active list from the mask words itself (a
// popcount scan of at most d_ff/32 words, read from L2), so there is no
// separate compaction launch between the predictor and this kernel.  The
// block's neurons are contiguous ranks of the list, balanced to within one
// neuron.  Their rows arrive through a ring of shared-memory stages filled by
// cp.async.bulk (the TMA engine's non-tensor copy: one instruction moves a
// whole 16-byte-aligned row, one mbarrier per stage counts the bytes), so each
// SM keeps several rows (tens of KB) in flight with no per-thread load
// registers.  Threads own fixed 16-byte column chunks: the up/gate dot products
// reduce across the block (warp shuffles + shared memory, one barrier per
// neuron), the down-projection accumulates in registers.  Per-block partial
// outputs are summed after a bounded grid barrier, each block reducing a
// column slice in a fixed order, so results are deterministic run to run.
#pragma once

#include "kernels.cuh"

namespace sffn {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;

// Bits of word w of the union of the B tokens' masks (or all neurons).
__device__ __forceinline__ uint32_t union_word(const GatherArgs& a, int w) {
  if (a.dense) {
    const int rem = a.f - w * 32;
    return rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
  }
  uint32_t u = 0;  // the mask is read-only while this kernel runs: the non-coherent path is safe
  for (int b = 0; b < a.B; ++b) u |= __ldg(&a.mask[(size_t)b * a.W + w]);
  return u;
}

template <typename T, int BT, int CPT>
__global__ void __launch_bounds__(kGatherThreads, 1) k_gather(const GatherArgs a) {
  constexpr int E = Chunk<T>::N;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_red[2][kGatherWarps][2 * BT];
  __shared__ int s_scan[kGatherWarps];
  __shared__ int s_total;
  __shared__ float4 s_rsum[kGatherThreads];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int B = a.B, d = a.d, W = a.W;
  const int NCH = d / E;
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const bool reglu = a.act == kReglu;
  const int nrows = reglu ? 3 : 2;
  const uint32_t stage_bytes = nrows * row_bytes;
  const int S = a.nstages;

  unsigned char* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + (size_t)S * stage_bytes);
  int32_t* list = reinterpret_cast<int32_t*>(bars + S);
  float* sbias = reinterpret_cast<float*>(list + a.list_cap);
  uint8_t* tokbits = reinterpret_cast<uint8_t*>(sbias + a.list_cap);

  // generation of this block's barrier flag, read before anyone can change it
  const uint32_t bar_gen = warp == 0 ? barrier_generation(a.bar_flags) : 0u;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }

  // ---- active list: exclusive scan of union popcounts, keep ranks [k0, k1)
  const int wpt = (W + kGatherThreads - 1) / kGatherThreads;
  const int w0 = tid * wpt;
  int cnt = 0;
  for (int k = 0; k < wpt; ++k)
    if (w0 + k < W) cnt += __popc(union_word(a, w0 + k));
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < kGatherWarps; ++w) {
      const int v = s_scan[w];
      s_scan[w] = run;
      run += v;
    }
    s_total = run;
  }
  __syncthreads();
  const int n_u = s_total;
  const int k0 = (int)((int64_t)n_u * cta / G);
  const int k1 = (int)((int64_t)n_u * (cta + 1) / G);
  const int nloc = k1 - k0;
  {
    int pos = s_scan[warp] + incl - cnt;
    for (int k = 0; k < wpt && pos < k1; ++k) {
      const int w = w0 + k;
      if (w >= W) break;
      uint32_t u = union_word(a, w);
      const int c = __popc(u);
      if (pos + c > k0) {
        uint32_t tw[4] = {0u, 0u, 0u, 0u};  // this word of each token's mask (B <= 4)
        for (int b = 0; b < B; ++b) tw[b] = a.dense ? 0xffffffffu : __ldg(&a.mask[(size_t)b * W + w]);
        while (u) {
          const int bit = __ffs(u) - 1;
          u &= u - 1;
          if (pos >= k0 && pos < k1) {
            list[pos - k0] = w * 32 + bit;
            uint32_t tb = 0;
            for (int b = 0; b < B; ++b) tb |= ((tw[b] >> bit) & 1u) << b;
            tokbits[pos - k0] = (uint8_t)tb;
          }
          ++pos;
        }
      } else {
        pos += c;
      }
    }
  }
  __syncthreads();
  for (int j = tid; j < nloc; j += kGatherThreads) sbias[j] = a.b != nullptr ? __ldg(&a.b[list[j]]) : 0.f;

  // ---- start the row pipeline
  const unsigned char* gup = static_cast<const unsigned char*>(a.w_up);
  const unsigned char* ggt = static_cast<const unsigned char*>(a.w_gate);
  const unsigned char* gdn = static_cast<const unsigned char*>(a.w_downT);
  uint64_t policy = 0;
  if (tid == 0) policy = policy_evict_first();
  auto issue = [&](int j) {
    const int s = j % S;
    const size_t off = (size_t)list[j] * a.wstride;
    unsigned char* dst = stages + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&bars[s], stage_bytes);
    bulk_g2s(dst, gup + off, row_bytes, &bars[s], policy);
    if (reglu) bulk_g2s(dst + row_bytes, ggt + off, row_bytes, &bars[s], policy);
    bulk_g2s(dst + (size_t)(nrows - 1) * row_bytes, gdn + off, row_bytes, &bars[s], policy);
  };
  if (tid == 0)
    for (int j = 0; j < min(S, nloc); ++j) issue(j);

  // ---- token values for this thread's column chunks
  float xr[BT][CPT][E];
  float yacc[BT][CPT][E];
  const T* xg = static_cast<const T*>(a.x);
#pragma unroll
  for (int bb = 0; bb < BT; ++bb)
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int ch = tid + c * kGatherThreads;
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (bb < B && ch < NCH) raw = *reinterpret_cast<const uint4*>(xg + (size_t)bb * d + ch * E);
      unpack<T>(raw, xr[bb][c]);
#pragma unroll
      for (int e = 0; e < E; ++e) yacc[bb][c][e] = 0.f;
    }

  // ---- one neuron per iteration
  int consumed = 0;
  bool failed = false;
  for (int j = 0; j < nloc; ++j) {
    const int s = j % S;
    const uint32_t par = (uint32_t)(j / S) & 1u;
    const bool ok = mbar_wait(&bars[s], par, a.hdr, a.wait_ns, 0x100u);
    const uint4* up = reinterpret_cast<const uint4*>(stages + (size_t)s * stage_bytes);
    const uint4* gt = up + NCH;
    const uint4* dn = up + (size_t)(nrows - 1) * NCH;

    float pu[BT], pg[BT];
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) pu[bb] = pg[bb] = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int ch = tid + c * kGatherThreads;
      if (ch < NCH) {
        float w[E];
        unpack<T>(up[ch], w);
#pragma unroll
        for (int bb = 0; bb < BT; ++bb)
#pragma unroll
          for (int e = 0; e < E; ++e) pu[bb] = fmaf(w[e], xr[bb][c][e], pu[bb]);
        if (reglu) {
          unpack<T>(gt[ch], w);
#pragma unroll
          for (int bb = 0; bb < BT; ++bb)
#pragma unroll
            for (int e = 0; e < E; ++e) pg[bb] = fmaf(w[e], xr[bb][c][e], pg[bb]);
        }
      }
    }
    float* rb = &s_red[j & 1][0][0];
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) {
      const float u = warp_sum(pu[bb]);
      const float g = reglu ? warp_sum(pg[bb]) : 0.f;
      if (lane == 0) {
        rb[warp * 2 * BT + bb] = u;
        rb[warp * 2 * BT + BT + bb] = g;
      }
    }
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    consumed = j + 1;
    // every thread has left iteration j-1, so its stage can be refilled
    if (tid == 0 && j >= 1 && j - 1 + S < nloc) issue(j - 1 + S);

    const uint32_t tb = tokbits[j];
    const float bias = sbias[j];  // written before the first barrier of the loop
    float act[BT];
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) {
      float u = 0.f, g = 0.f;
#pragma unroll
      for (int w = 0; w < kGatherWarps; ++w) {
        u += rb[w * 2 * BT + bb];
        g += rb[w * 2 * BT + BT + bb];
      }
      const float v = reglu ? fmaxf(g + bias, 0.f) * u : fmaxf(u + bias, 0.f);
      act[bb] = ((tb >> bb) & 1u) ? v : 0.f;
    }
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int ch = tid + c * kGatherThreads;
      if (ch < NCH) {
        float w[E];
        unpack<T>(dn[ch], w);
#pragma unroll
        for (int bb = 0; bb < BT; ++bb)
          if (act[bb] != 0.f) {
#pragma unroll
            for (int e = 0; e < E; ++e) yacc[bb][c][e] = fmaf(act[bb], w[e], yacc[bb][c][e]);
          }
      }
    }
  }
  if (failed) {
    // let the copies already issued land before the block exits (bounded)
    if (tid == 0) {
      const int issued = consumed == 0 ? min(S, nloc) : min(nloc, consumed - 1 + S);
      for (int j = consumed; j < issued; ++j)
        mbar_wait(&bars[j % S], (uint32_t)(j / S) & 1u, a.hdr, a.wait_ns, 0x101u);
    }
    return;
  }

  // ---- per-block partial, then the cross-block column reduction
  float* dst = G == 1 ? a.y : a.y_part + (size_t)cta * B * d;
#pragma unroll
  for (int bb = 0; bb < BT; ++bb)
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int ch = tid + c * kGatherThreads;
      if (bb < B && ch < NCH) {
        float4* o = reinterpret_cast<float4*>(dst + (size_t)bb * d + ch * E);
#pragma unroll
        for (int e = 0; e < E; e += 4)
          o[e / 4] = make_float4(yacc[bb][c][e], yacc[bb][c][e + 1], yacc[bb][c][e + 2], yacc[bb][c][e + 3]);
      }
    }
  if (G == 1) return;
  if (!grid_barrier(a.hdr, a.bar_flags, (uint32_t)G, bar_gen, a.wait_ns, 0x200u)) return;

  const int N4 = B * d / 4;
  const float4* yp4 = reinterpret_cast<const float4*>(a.y_part);
  float4* y4 = reinterpret_cast<float4*>(a.y);
  const int q0 = (int)((int64_t)N4 * cta / G), q1 = (int)((int64_t)N4 * (cta + 1) / G);
  for (int qb = q0; qb < q1; qb += kGatherThreads) {
    const int nq = min(kGatherThreads, q1 - qb);
    const int GS = max(1, min(G, kGatherThreads / nq));
    if (tid < nq * GS) {
      const int qi = tid % nq, gs = tid / nq;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int g = gs; g < G; g += GS) {
        const float4 v = __ldcg(&yp4[(size_t)g * N4 + qb + qi]);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      s_rsum[gs * nq + qi] = acc;
    }
    __syncthreads();
    if (tid < nq) {
      float4 t = s_rsum[tid];
      for (int gs = 1; gs < GS; ++gs) {
        const float4 v = s_rsum[gs * nq + tid];
        t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
      }
      y4[qb + tid] = t;
    }
    __syncthreads();
  }
}

template <typename T, int BT, int CPT>
cudaError_t gather_launch(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_gather<T, BT, CPT>, cfg.smem, &cur);
  if (e != cudaSuccess) return e;
  k_gather<T, BT, CPT><<<grid, kGatherThreads, cfg.smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int CPT>
cudaError_t gather_bt(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  constexpr int E = Chunk<T>::N;
  if (cfg.bt == 1) return gather_launch<T, 1, CPT>(cfg, a, grid, s);
  if constexpr (2 * CPT * E <= 64)
    if (cfg.bt == 2) return gather_launch<T, 2, CPT>(cfg, a, grid, s);
  if constexpr (4 * CPT * E <= 64)
    if (cfg.bt == 4) return gather_launch<T, 4, CPT>(cfg, a, grid, s);
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t gather_dispatch(const GatherConfig& cfg, const GatherArgs& a, int grid, cudaStream_t s) {
  switch (cfg.cpt) {
    case 1: return gather_bt<T, 1>(cfg, a, grid, s);
    case 2: return gather_bt<T, 2>(cfg, a, grid, s);
    case 3: return gather_bt<T, 3>(cfg, a, grid, s);
    case 4: return gather_bt<T, 4>(cfg, a, grid, s);
    case 6: return gather_bt<T, 6>(cfg, a, grid, s);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace sffn
