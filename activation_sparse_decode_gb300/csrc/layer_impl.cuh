// One decode token through one FFN layer in a single launch: predictor,
// threshold, neuron-aware row gather, activation and down projection.
//
// Why one kernel.  At batch 1 a layer moves only tens of MB, a few microseconds
// of HBM time, so the cost of separate launches and of their dependency gaps is
// as large as the work.  Here every block works through all phases, and the
// only grid-wide dependency is the predictor's hidden layer: block c reduces
// the rows k = c, c + G, ... of h = V x over all of d and publishes each in a
// tagged workspace slot; every block then acquires all r slots (bounded
// polling), which also orders every block's zeroed output slices before the
// accumulation.
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
// Overlap.  Under programmatic dependent launch the kernel warms L2 with its
// V rows, U rows (when it stages them), biases, hot rows and the LayerNorm's
// inputs while the previous kernel finishes; its first V rows go to
// registers, its U rows and biases to shared memory, and its hot rows -- the
// first owned neurons, almost always active -- to the first ring stages before
// the predictor has decided (before the wait, or right behind the LayerNorm's
// loads when the token is formed from the previous layer).  The active rows stream through a ring of
// one-neuron stages filled by per-thread 16-byte cp.async (each thread copies
// the chunks it later reads), and the block's partial output is added into y
// with vector float atomics, so there is no second grid-wide step.
//
// Stacked layers: when y_prev is given, the block first forms this layer's
// input x = round(LayerNorm(x_prev + y_prev)) itself (every block computes the
// same values; each writes its slice of the stored result), so no separate
// LayerNorm launch sits between layers.
#pragma once

#include "kernels.cuh"

namespace sffn {

// Phase timestamps for profiling builds (compiled out unless SFFN_PHASE_TRACE
// is defined, in which case the including file provides sffn_phase_trace()).
#ifdef SFFN_PHASE_TRACE
#define SFFN_TRACE(k) sffn_phase_trace(k)
#define SFFN_TRACE_VAL(k, v) sffn_phase_value(k, v)
#define SFFN_TRACE_AT(k, t) sffn_phase_trace_at(k, t)
#define SFFN_TRACE_GROUP(k) sffn_phase_trace_group(k)
#else
#define SFFN_TRACE_GROUP(k) ((void)0)
#define SFFN_TRACE_AT(k, t) ((void)0)
#define SFFN_TRACE(k) ((void)0)
#define SFFN_TRACE_VAL(k, v) ((void)0)
#endif

constexpr int kLayerThreads = 256;
constexpr int kLayerWarps = kLayerThreads / 32;
constexpr int kGroup = 2;  // neurons per block-wide reduction in the row ring
constexpr int kSlotStride = 16;  // launch slots: one per 128-byte line (16 words)
// The thread that publishes the balancing exchange's count (its fence waits
// for its own copies in flight).
constexpr int kBarrierThread = kLayerThreads - 32;

// The ring's stage wait once the first test has failed: kept out of line so
// that the loop body stays small enough for the instruction cache.
static __device__ __noinline__ bool pair_wait_slow(uint64_t* bar, WsHeader* h, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      set_status(h, kStTimeout, 0x307u);
      return false;
    }
  }
  return true;
}

static __device__ __noinline__ bool layer_wait_slow(uint64_t* bar, uint32_t parity, WsHeader* h, uint64_t limit_ns) {
  return mbar_wait(bar, parity, h, limit_ns, 0x303u);
}

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

// One 16-byte chunk of values rounded to the stored format (round to nearest even).
template <typename T>
__device__ __forceinline__ uint4 pack_chunk(const float* v);
template <>
__device__ __forceinline__ uint4 pack_chunk<float>(const float* v) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
template <>
__device__ __forceinline__ uint4 pack_chunk<__half>(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 pack_chunk<__nv_bfloat16>(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The forms up to three chunks (d_model up to 6144 for 16-bit weights) are
// held to two blocks per SM worth of registers (128): uncapped the three-chunk
// form needs 139, and the OPT-13B-shaped layer then runs one block per SM,
// 2.4% slower.  The larger forms run one block per SM.
template <typename T, int CPT, int ACT>
__global__ void __launch_bounds__(kLayerThreads, CPT <= 3 ? 2 : 1) k_layer(const LayerArgs a) {
  constexpr int CPL = 4;  // up to 4 16-byte chunks of a U row per lane (rank <= 128 * elements per chunk)
  constexpr int E = Chunk<T>::N;
  constexpr int ES = sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_red[2][kLayerWarps][kGroup][2];
  __shared__ float s_warp[kLayerWarps];
  __shared__ int s_nloc;
  __shared__ int s_passed;
  __shared__ __align__(8) uint64_t s_xbar;  // pair exchange: the partner's message has landed
  __shared__ int s_pcnt;                    // pair exchange: the partner's row count

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int d = a.d, f = a.f, r = a.r;
  const int NCH = d / E;       // 16-byte chunks per d-row
  const int NC = r / E;        // 16-byte chunks per U row
  const uint32_t row_bytes = (uint32_t)d * ES;
  const uint32_t urow_bytes = (uint32_t)r * ES;
  constexpr bool reglu = ACT == kReglu;
  constexpr int nrows = reglu ? 3 : 2;
  const uint32_t stage_bytes = nrows * row_bytes;
  const int S = a.nstages;
  const int n_own = c < f ? (f - c + G - 1) / G : 0;
  const int own_cap = (f + G - 1) / G;
  const int nwords = (own_cap + 31) / 32;
  // look-ahead: this call's rows from la_in, the predictor (the next layer's)
  // into la_out; predict-only: the predictor into la_out and nothing else
  const bool lookahead = a.la_in != nullptr;
  const bool ponly = a.predict_only != 0;
  uint32_t* const sc_out = (lookahead || ponly) ? a.la_out : a.mask;  // mask words the scores set

  // ---- shared memory carve-up (offsets are multiples of 16)
  unsigned char* region = smem;  // U rows (phases 0-4), then the row ring
  float* hs = reinterpret_cast<float*>(smem + a.region_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(hs + ((r + 3) & ~3));
  float* ownb = reinterpret_cast<float*>(bars + S + 1);
  float* ownpb = ownb + own_cap;
  uint32_t* words = reinterpret_cast<uint32_t*>(ownpb + own_cap);
  int32_t* list = reinterpret_cast<int32_t*>(words + nwords);  // active neurons (global index) per ring position
  float* lbias = reinterpret_cast<float*>(list + own_cap);       // their biases
  uint8_t* s_act = reinterpret_cast<uint8_t*>(lbias + own_cap);  // predicted-active flag per owned row
  // pair exchange inbox {neuron, bias bits}: 8-byte entries, so 16-byte aligned
  int2* inbox = reinterpret_cast<int2*>((reinterpret_cast<uintptr_t>(s_act + own_cap) + 15) & ~uintptr_t(15));
  // balancing scratch, last: allocated only for launches that balance
  int32_t* bal_cnt = reinterpret_cast<int32_t*>(inbox + ((own_cap + 1) & ~1));  // rows per block,
  int32_t* bal_keep = bal_cnt + G;                                                // rows each block keeps,
  int32_t* bal_einc = bal_keep + G;  // inclusive prefix of given-away rows
  SFFN_TRACE(0);

  const unsigned char* gup = static_cast<const unsigned char*>(a.w_up);
  const unsigned char* ggt = static_cast<const unsigned char*>(a.w_gate);
  const unsigned char* gdn = static_cast<const unsigned char*>(a.w_downT);
  // Owned row j into stage s: every thread copies its own 16-byte chunks (the
  // same chunks it later reads, so no thread waits on another's data) and
  // arrives on the stage barrier when they have landed.  Expected arrivals per
  // phase: one per thread.
  auto fill = [&](int s, int neuron) {
    const size_t off = (size_t)neuron * a.wstride;
    unsigned char* dst = region + (size_t)s * stage_bytes;
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      if (ch < NCH) {
        cp_async16(dst + (size_t)ch * 16, gup + off + (size_t)ch * 16);
        if (reglu) cp_async16(dst + row_bytes + (size_t)ch * 16, ggt + off + (size_t)ch * 16);
        cp_async16(dst + (size_t)(nrows - 1) * row_bytes + (size_t)ch * 16, gdn + off + (size_t)ch * 16);
      }
    }
    cp_async_arrive_noinc(&bars[s]);
  };

  // ---- phase 0a: before the previous kernel on the stream has finished
  // (programmatic dependent launch) the kernel touches only its own shared
  // memory and warms L2: this block's V rows, owned U rows and biases, hot
  // rows and warm rows are prefetched into L2.  A prefetch of a line that
  // kernel is still writing is harmless (the later reads see its writes).
  // The weights themselves are read here only when the layer declares them
  // static (no kernel writes them while the layer exists): then the first V
  // rows go to registers, the owned U rows and biases to shared memory and
  // the hot rows to the first ring stages before the wait.  The token, the
  // outputs and the workspace may still be in use by that kernel.
  uint64_t* ubar = bars + S;  // completes when this block's U rows and biases have landed
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], kLayerThreads);
    mbar_init(ubar, kLayerThreads);
    if (a.cluster == 2) mbar_init(&s_xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Pair exchange barrier sequence (clusters of two; every path takes it):
  // phase 1 arrives here and is waited before this block first writes into
  // its partner's shared memory, so the partner's barrier is initialised;
  // phase 2 arrives after the last such write and is waited just before the
  // block exits, so no block leaves while its partner may still write to it.
  if (a.cluster == 2) cluster_arrive();
  // An early exit still sends the partner a count of zero (it does not wait
  // for this block's rows) and passes both phases.
  auto pair_exit_early = [&]() {
    cluster_wait();
    if (tid == 0) {
      const uint32_t peer = cluster_rank() ^ 1u;
      st_peer_s32(peer_smem(&s_pcnt, peer), 0);
      mbar_arrive_remote(peer_smem(&s_xbar, peer));
    }
    cluster_arrive();
    cluster_wait();
  };
  // Once this block has sent its rows to the partner (look-ahead sends them
  // early), an exit only passes phase 2.
  bool pair_sent = false;
  auto pair_exit = [&]() {
    if (!pair_sent) {
      pair_exit_early();
    } else {
      cluster_arrive();
      cluster_wait();
    }
  };
  const int nh = c < r ? (r - c + G - 1) / G : 0;  // h rows of this block: c, c + G, ...
  const uint4* V4 = static_cast<const uint4*>(a.V);
  const unsigned char* Ub = static_cast<const unsigned char*>(a.U);
  const int n_hot = !ponly && c < a.hot_rows ? min(a.hot_stages, min(n_own, (a.hot_rows - c + G - 1) / G)) : 0;
  {
    if (tid < nh) bulk_prefetch_l2(V4 + (size_t)(c + tid * G) * NCH, row_bytes);
    for (int j = tid; j < n_own; j += kLayerThreads) {
      if (a.b != nullptr) prefetch_l2(&a.b[c + j * G]);
      prefetch_l2(&a.pb[c + j * G]);
    }
    // (U rows too many to stage are not warmed: the scores stream them once,
    // and 100 MB of prefetches queued ahead of the token's loads cost more
    // than they saved -- 81.9 against 81.5 us per layer on the OPT-175B shape)
    const int ulines = a.u_smem ? (urow_bytes + 127) / 128 : 0;
    for (int q = tid; q < n_own * ulines; q += kLayerThreads) {
      const int j = q / ulines, l = q - j * ulines;
      prefetch_l2(Ub + (size_t)(c + (size_t)j * G) * urow_bytes + l * 128);
    }
    // the LayerNorm's gamma and beta, and the previous layer's token (which
    // that kernel wrote at its start): every block reads all of them right
    // after the wait, so each block warms every G-th line of them
    if (a.y_prev != nullptr) {
      const int glines = (d * 4 + 127) / 128;
      for (int l = c + tid * G; l < glines; l += kLayerThreads * G) {
        if (a.ln_gamma != nullptr) prefetch_l2(reinterpret_cast<const char*>(a.ln_gamma) + (size_t)l * 128);
        if (a.ln_beta != nullptr) prefetch_l2(reinterpret_cast<const char*>(a.ln_beta) + (size_t)l * 128);
      }
      const int xlines = (int)((row_bytes + 127) / 128);
      for (int l = c + tid * G; l < xlines; l += kLayerThreads * G)
        prefetch_l2(static_cast<const char*>(a.x) + (size_t)l * 128);
    }
    const int nw = !ponly && c < a.warm_rows ? min(n_own, (a.warm_rows - c + G - 1) / G) : 0;
    const int rlines = (row_bytes + 127) / 128;
    for (int q = tid; q < max(n_hot, nw) * rlines; q += kLayerThreads) {
      const int j = q / rlines, l = q - j * rlines;
      const size_t off = (size_t)(c + (size_t)j * G) * a.wstride + (size_t)l * 128;
      prefetch_l2(gup + off);
      if (reglu) prefetch_l2(ggt + off);
      prefetch_l2(gdn + off);
    }
  }
  // Staging of this block's weights: the first V rows (registers, RB rows
  // per batch, every load of a batch in flight at once), owned biases and U
  // rows (shared memory, completing on ubar) and hot rows (the first ring
  // stages).
  constexpr int RB = CPT <= 2 ? 1 : CPT <= 3 ? 2 : 4;
  uint4 vr[RB][CPT];
  auto stage_weights = [&]() {
#pragma unroll
    for (int jj = 0; jj < RB; ++jj)
#pragma unroll
      for (int cq = 0; cq < CPT; ++cq) {
        const int ch = tid + cq * kLayerThreads;
        vr[jj][cq] = jj < nh && ch < NCH ? ldg_stream(V4 + (size_t)(c + jj * G) * NCH + ch) : make_uint4(0, 0, 0, 0);
      }
    for (int j = tid; j < n_own; j += kLayerThreads) {
      const int i = c + j * G;
      if (!lookahead) {  // look-ahead loads them with the mask bits, before the list
        if (a.b != nullptr)
          cp_async4(&ownb[j], &a.b[i]);
        else
          ownb[j] = 0.f;
      }
      cp_async4(&ownpb[j], &a.pb[i]);
    }
    if (a.u_smem)  // owned U rows -> shared memory, 16 bytes per copy
      for (int q = tid; q < n_own * NC; q += kLayerThreads) {
        const int j = q / NC, ch = q - j * NC;
        cp_async16(region + a.u_off + (size_t)j * urow_bytes + ch * 16,
                   Ub + (size_t)(c + (size_t)j * G) * urow_bytes + ch * 16);
      }
    cp_async_arrive_noinc(ubar);
  };
  // the hot rows into the first ring stages (with a token formed by the
  // LayerNorm, after that token's loads, which every later phase waits for:
  // 80.4 against 80.5 us per layer on the OPT-175B-shaped stack)
  auto fill_hot = [&]() {
    for (int j = 0; j < n_hot; ++j) fill(j, c + j * G);
  };
  // hot rows: before the wait when the token is a plain input; behind the
  // LayerNorm's loads when it is formed from the previous layer
  if (a.static_weights) {
    stage_weights();
    if (a.y_prev == nullptr) fill_hot();
  }
  grid_dependency_wait();       // the previous kernel has completed and its writes are visible
  grid_dependents_launch();     // the next one may start its phase 0a
  SFFN_TRACE(18);

  // ---- the token's loads first (to registers: nothing below waits for
  // them), then, unless staged above, this block's weights.
  uint4 xreg[CPT];
  if (a.y_prev == nullptr) {
    const uint4* xg = static_cast<const uint4*>(a.x);
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      xreg[cq] = ch < NCH ? __ldcg(xg + ch) : make_uint4(0, 0, 0, 0);
    }
  }
  if (!a.static_weights) {
    stage_weights();
    if (a.y_prev == nullptr) fill_hot();
  }


  // ---- phase 0b: this launch's tag, the token, zeroed outputs.
  // Tag: every block adds one to the workspace's launch counter; the last
  // arrival of a launch rounds the counter up to the next multiple of 2^20,
  // so the counter's high part numbers the launches whatever their grid
  // sizes, and every block reads the same number from its own arrival.
  __shared__ uint32_t s_tag;
  if (tid == kLayerThreads - 32) {
    unsigned long long old;
    asm volatile("atom.add.relaxed.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(&a.hdr->arrivals) : "memory");
    const unsigned long long base = old & ~((1ull << 20) - 1ull);
    if (old - base == (unsigned long long)(G - 1))
      asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(&a.hdr->arrivals),
                   "l"((unsigned long long)((1u << 20) - G))
                   : "memory");
    s_tag = (uint32_t)(base >> 20) + 1u;  // never 0, the value of a zeroed slot
  }
  // outputs zeroed by the h-row owners, slice k of y and of the mask with h
  // row k, so that the slots every block acquires below cover all of them
  for (int j = 0; j < nh; ++j) {
    const int k = c + j * G;
    if (a.y != nullptr) {
      float4* y4 = reinterpret_cast<float4*>(a.y);
      const int N4 = d / 4;
      const int q1 = (int)((int64_t)N4 * (k + 1) / r);
      for (int q = (int)((int64_t)N4 * k / r) + tid; q < q1; q += kLayerThreads) y4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sc_out != nullptr) {
      const int W = (f + 31) / 32;
      const int w1 = (int)((int64_t)W * (k + 1) / r);
      for (int w = (int)((int64_t)W * k / r) + tid; w < w1; w += kLayerThreads) sc_out[w] = 0u;
    }
  }
  // The token: loaded, or formed from the previous layer by residual +
  // LayerNorm.  Thread tid only ever uses chunks tid, tid + 256, ... of it
  // (the h rows and the ring read the same chunks of every row), so it stays
  // in registers, packed in the stored format (xpk), and no shared memory
  // holds it.
  uint4 xpk[CPT];
  if (a.y_prev == nullptr) {
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) xpk[cq] = xreg[cq];
  } else {
    // x_prev + y_prev is read once into registers (every chunk's loads in
    // flight together); mean and biased variance by two block sums over them
    const T* xp = static_cast<const T*>(a.x);
    uint4 xr[CPT];
    float4 yr[CPT][E / 4];
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      xr[cq] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e4 = 0; e4 < E / 4; ++e4) yr[cq][e4] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ch < NCH) {
        xr[cq] = __ldcg(reinterpret_cast<const uint4*>(xp + ch * E));
        const float4* yp = reinterpret_cast<const float4*>(a.y_prev + ch * E);
#pragma unroll
        for (int e4 = 0; e4 < E / 4; ++e4) yr[cq][e4] = __ldcg(&yp[e4]);
      }
    }
    fill_hot();
    float v[CPT][E];
    float s = 0.f;
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      unpack<T>(xr[cq], v[cq]);
#pragma unroll
      for (int e4 = 0; e4 < E / 4; ++e4) {
        v[cq][4 * e4] += yr[cq][e4].x;
        v[cq][4 * e4 + 1] += yr[cq][e4].y;
        v[cq][4 * e4 + 2] += yr[cq][e4].z;
        v[cq][4 * e4 + 3] += yr[cq][e4].w;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) s += v[cq][e];
    }
    const float mean = layer_block_sum(s, s_warp) / (float)d;
    SFFN_TRACE(20);
    float q = 0.f;
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq)
      if (tid + cq * kLayerThreads < NCH)
#pragma unroll
        for (int e = 0; e < E; ++e) q = fmaf(v[cq][e] - mean, v[cq][e] - mean, q);
    const float var = layer_block_sum(q, s_warp) / (float)d;
    const float rstd = 1.0f / sqrtf(var + a.ln_eps);
    SFFN_TRACE(21);
#pragma unroll
    for (int cq = 0; cq < CPT; ++cq) {
      const int ch = tid + cq * kLayerThreads;
      if (ch < NCH) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float o = (v[cq][e] - mean) * rstd;
          if (a.ln_gamma != nullptr) o *= a.ln_gamma[ch * E + e];
          if (a.ln_beta != nullptr) o += a.ln_beta[ch * E + e];
          v[cq][e] = o;
        }
      }
      xpk[cq] = ch < NCH ? pack_chunk<T>(v[cq]) : make_uint4(0, 0, 0, 0);
    }
    if (a.x_ln_out != nullptr) {  // chunk ch of the new x is stored by block ch mod G
      uint4* xo = static_cast<uint4*>(a.x_ln_out);
#pragma unroll
      for (int cq = 0; cq < CPT; ++cq) {
        const int ch = tid + cq * kLayerThreads;
        if (ch < NCH && ch % G == c) xo[ch] = xpk[cq];
      }
    }
    SFFN_TRACE(22);
  }
  __syncthreads();

  // ---- the ring's list and its first fills (start_ring), and the pair split
  // (settle_ring).  Normal calls run both after the scores; look-ahead calls
  // run start_ring as soon as the token is formed (their rows are known from
  // la_in) and settle_ring after the predictor.
  //
  // The list: positions 0..n_hot-1 are the prefetched rows, active or not (an
  // inactive one carries the bias -inf, which the activation below turns into
  // an exact zero: it adds nothing), then the other active owned rows in
  // ascending order.  Warp 0 takes one 32-row word per step, lane k holding
  // row k's flag; a ballot forms the word and each active lane writes its row
  // at its rank.
  //
  // Pair exchange (clusters of two blocks): a token's active rows fall
  // unevenly on the blocks, and the block with the most sets the kernel's
  // length.  The two blocks of a cluster split their rows evenly -- T rows
  // in all, capacities ceil(T/2) (rank 0) and floor(T/2), each keeping its
  // own rows up to max(capacity, prefetched stages) and handing the rest,
  // its last rows, to the other -- without waiting for each other: each
  // block keeps at least k_safe = max(count/2, prefetched stages) rows
  // whatever the partner has, streams those at once, and sends its count and
  // rows [k_safe, count) into the partner's inbox (shared-memory stores, then
  // one release-arrive on the partner's barrier).  The split is settled when
  // the partner's message is in, from this block's own shared memory.
  //
  // The rows fetched in phase 0 are list positions 0..n_hot-1, in their
  // stages already.  List position p uses stage p % S.  Own rows start
  // streaming at once, up to the prefill count when the rows are balanced
  // afterwards (every block keeps at least that many of its own; traffic in
  // flight lengthens the balancing exchange's round trips, so it runs with
  // the request queues short).
  const int P = a.hot_stages;
  // ring stages that do not overlap the staged U rows: the only ones a
  // look-ahead call may fill before the scores are done
  const int free_stages = a.u_smem ? min(S, (int)(a.u_off / stage_bytes)) : S;
  const int early = lookahead ? free_stages : S;
  int nloc = 0, k_safe = 0, pre = 0;
  auto start_ring = [&]() {
    if (warp == 0) {
      for (int j = lane; j < n_hot; j += 32) {
        list[j] = c + j * G;
        lbias[j] = s_act[j] != 0 ? ownb[j] : -INFINITY;
      }
      int base = n_hot;
      for (int q = 0; q < nwords; ++q) {
        const int j = q * 32 + lane;
        const bool on = j >= n_hot && j < n_own && s_act[j] != 0;
        const uint32_t bits = __ballot_sync(0xffffffffu, on);
        if (on) {
          const int pos = base + __popc(bits & ((1u << lane) - 1u));
          list[pos] = c + j * G;
          lbias[pos] = ownb[j];
        }
        base += __popc(bits);
      }
      if (lane == 0) s_nloc = base;
    }
    __syncthreads();
    nloc = s_nloc;
    SFFN_TRACE_VAL(11, nloc);
    k_safe = nloc;
    if (a.cluster == 2) {
      k_safe = min(nloc, max(nloc / 2, a.hot_stages));
      cluster_wait();  // phase 1: the partner's barrier is initialised
      const uint32_t peer = cluster_rank() ^ 1u;
      for (int t = tid; t < nloc - k_safe; t += kLayerThreads)
        st_peer_v2(peer_smem(inbox + t, peer), list[k_safe + t], __float_as_int(lbias[k_safe + t]));
      __syncthreads();  // every entry is stored before the release below
      if (tid == 0) {
        st_peer_s32(peer_smem(&s_pcnt, peer), nloc);
        mbar_arrive_remote(peer_smem(&s_xbar, peer));
      }
      pair_sent = true;
    }
    SFFN_TRACE(5);
    pre = a.balance ? min(nloc, P) : k_safe;
    for (int p = n_hot; p < min(early, pre); ++p) fill(p % S, list[p]);
  };
  // false: the partner's message never came (status set); the caller returns
  auto settle_ring = [&]() -> bool {
    // the stages a look-ahead call could not fill before the scores
    for (int p = max(n_hot, min(early, pre)); p < min(S, pre); ++p) fill(p % S, list[p]);
    if (a.cluster != 2) return true;
    bool got = mbar_try_wait_cluster(&s_xbar, 0);
    if (!got) got = pair_wait_slow(&s_xbar, a.hdr, a.wait_ns);
    if (__syncthreads_or(!got)) {
      cp_async_wait_all();
      cluster_arrive();
      cluster_wait();
      return false;
    }
    const int rk = (int)cluster_rank();
    const int np = s_pcnt;
    const int tot = nloc + np;
    const int cap_me = rk == 0 ? (tot + 1) / 2 : tot / 2, cap_peer = tot - cap_me;
    const int keep_peer = min(np, max(cap_peer, P));
    if (np > keep_peer) {  // the partner's rows [keep_peer, np), from the inbox
      const int ks_peer = min(np, max(np / 2, P));
      for (int t = tid; t < np - keep_peer; t += kLayerThreads) {
        const int2 e = inbox[keep_peer - ks_peer + t];
        list[nloc + t] = e.x;
        lbias[nloc + t] = __int_as_float(e.y);
      }
      nloc += np - keep_peer;
    } else {
      nloc = min(nloc, max(cap_me, P));
    }
    __syncthreads();  // the received entries are in place for every thread
    cluster_arrive();  // phase 2: no more writes into the partner's shared memory
    for (int p = max(n_hot, min(S, k_safe)); p < min(S, nloc); ++p) fill(p % S, list[p]);
    SFFN_TRACE(16);
    return true;
  };

  // Look-ahead: this call's active rows are already decided (la_in, written
  // by the previous call); their biases are read here with them, and the ring
  // starts before the predictor of the next layer runs.
  if (lookahead) {
    for (int j = tid; j < n_own; j += kLayerThreads) {
      const int i = c + j * G;
      s_act[j] = (uint8_t)((__ldcg(a.la_in + (i >> 5)) >> (i & 31)) & 1u);
      ownb[j] = a.b != nullptr ? __ldg(a.b + i) : 0.f;
    }
    __syncthreads();
    start_ring();
  }

  SFFN_TRACE(1);
  // ---- phase 1: this block's h rows, h_k = V_k . x in fp32 (each a fixed-
  // order block reduction), published with the tag in slot k (one 128-byte
  // line per slot, so that the polls below spread over L2).  Each slot is one
  // release store after the whole block's writes above (the zeroed slices).
  const uint32_t tag = s_tag;
  unsigned long long* slots = a.h_slots;
  __shared__ float s_hred[kLayerWarps][RB];
  for (int j0 = 0; j0 < nh; j0 += RB) {
    if (j0 > 0)
#pragma unroll
      for (int jj = 0; jj < RB; ++jj)
#pragma unroll
        for (int cq = 0; cq < CPT; ++cq) {
          const int ch = tid + cq * kLayerThreads;
          if (j0 + jj < nh && ch < NCH) vr[jj][cq] = ldg_stream(V4 + (size_t)(c + (j0 + jj) * G) * NCH + ch);
        }
    float acc[RB];
#pragma unroll
    for (int jj = 0; jj < RB; ++jj) {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int cq = 0; cq < CPT; ++cq) {
        const int ch = tid + cq * kLayerThreads;
        if (j0 + jj < nh && ch < NCH) {
          float w[E], xv[E];
          unpack<T>(vr[jj][cq], w);
          unpack<T>(xpk[cq], xv);
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            acc0 = fmaf(w[e], xv[e], acc0);
            acc1 = fmaf(w[e + 1], xv[e + 1], acc1);
          }
        }
      }
      acc[jj] = warp_sum(acc0 + acc1);
    }
    __syncthreads();  // the previous batch's sums have been read
    if (lane == 0)
#pragma unroll
      for (int jj = 0; jj < RB; ++jj) s_hred[warp][jj] = acc[jj];
    __syncthreads();
    if (tid < RB && j0 + tid < nh) {
      float hk = 0.f;
#pragma unroll
      for (int w = 0; w < kLayerWarps; ++w) hk += s_hred[w][tid];
      asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(slots + (size_t)(c + (j0 + tid) * G) * kSlotStride),
                   "l"(((unsigned long long)tag << 32) | __float_as_uint(hk))
                   : "memory");
    }
  }
  SFFN_TRACE(2);

  // ---- phase 2: every h slot of this launch: h is complete and every
  // block's zeroed slices precede what follows.  Warp 0 polls, lane l slots
  // l, l + 32, ..., with relaxed loads (each round's loads all in flight, a
  // short pause between rounds), then one acquire fence.
  bool ok = true;
  if (warp == 0) {
    uint32_t pending = 0;  // bit q: slot lane + 32 q not yet tagged
    for (int q = 0; q < 32; ++q)
      if (lane + 32 * q < r) pending |= 1u << q;
    uint64_t t0 = 0;
    const int nq = (r - lane + 31) / 32;  // this lane's slots
    while (true) {
      // batches of PB slots, statically indexed so that the values stay in
      // registers and every load of a batch is in flight before any check
      // (the wide forms poll up to 1024 slots: all of a lane's 32 at once)
      constexpr int PB = CPT >= 4 ? 32 : 16;
      for (int q0 = 0; q0 < nq; q0 += PB) {
        unsigned long long v[PB];
#pragma unroll
        for (int u = 0; u < PB; ++u) {
          v[u] = 0ull;
          if (q0 + u < nq && ((pending >> (q0 + u)) & 1u))
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];"
                         : "=l"(v[u])
                         : "l"(slots + (size_t)(lane + 32 * (q0 + u)) * kSlotStride)
                         : "memory");
        }
#pragma unroll
        for (int u = 0; u < PB; ++u)
          if (q0 + u < nq && ((pending >> (q0 + u)) & 1u) && (uint32_t)(v[u] >> 32) == tag) {
            hs[lane + 32 * (q0 + u)] = __uint_as_float((uint32_t)v[u]);
            pending &= ~(1u << (q0 + u));
          }
      }
      if (!__any_sync(0xffffffffu, pending != 0)) break;
      if (t0 == 0) t0 = globaltimer_ns();
      if (globaltimer_ns() - t0 > a.wait_ns) {
        if (pending) set_status(a.hdr, kStTimeout, 0x300u);
        ok = false;
        break;
      }
      __nanosleep(64);
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
  }
  const bool passed = !__syncthreads_or(!ok);
  SFFN_TRACE_AT(13, 0);
  if (!passed) {
    cp_async_wait_all();  // nothing of this block is left in flight
    if (a.cluster == 2) pair_exit();
    return;
  }
  SFFN_TRACE(3);

  // ---- phase 4: scores of the owned neurons.  One warp per 32-row word: lane
  // l holds 16-byte chunks l, l+32, ... of every row, rows are summed with a
  // warp all-reduce, and lane k keeps row k's score.  A compact loop: fully
  // unrolled variants of it overflow the instruction cache.
  SFFN_TRACE(4);
  // this block's U rows and biases have landed (every thread's copies)
  if (!mbar_try_wait(ubar, 0) && !layer_wait_slow(ubar, 0, a.hdr, a.wait_ns)) ok = false;
  if (__syncthreads_or(!ok)) {
    cp_async_wait_all();
    if (a.cluster == 2) pair_exit();
    return;
  }
  SFFN_TRACE(8);
  if (a.u_smem) {
    // Lr lanes per row from shared memory (a power of two, as many as keep all
    // threads busy); each group starts at a row-dependent chunk so the lanes of
    // one shared-memory phase hit distinct banks.
    int Lr = 1;
    while (Lr < 32 && 2 * Lr <= NC && n_own * 2 * Lr <= kLayerThreads) Lr *= 2;
    const int rows_per_pass = kLayerThreads / Lr;
    const int sub = tid % Lr;
    for (int j0 = 0; j0 < n_own; j0 += rows_per_pass) {
      const int j = j0 + tid / Lr;
      float acc0 = 0.f, acc1 = 0.f;
      if (j < n_own) {
        const uint4* row = reinterpret_cast<const uint4*>(region + a.u_off + (size_t)j * urow_bytes);
        const int rot = (j * Lr) & 7;
        for (int k = sub; k < NC; k += Lr) {
          int ch = k + rot;
          if (ch >= NC) ch -= NC;
          if (ch >= NC) ch %= NC;
          float w[E];
          unpack<T>(row[ch], w);
          const float4* hp = reinterpret_cast<const float4*>(hs + ch * E);
          const float4 h0 = hp[0];
          acc0 = fmaf(w[0], h0.x, acc0);
          acc1 = fmaf(w[1], h0.y, acc1);
          acc0 = fmaf(w[2], h0.z, acc0);
          acc1 = fmaf(w[3], h0.w, acc1);
          if (E > 4) {
            const float4 h1 = hp[1];
            acc0 = fmaf(w[E > 4 ? 4 : 0], h1.x, acc0);
            acc1 = fmaf(w[E > 4 ? 5 : 0], h1.y, acc1);
            acc0 = fmaf(w[E > 4 ? 6 : 0], h1.z, acc0);
            acc1 = fmaf(w[E > 4 ? 7 : 0], h1.w, acc1);
          }
        }
      }
      float acc = acc0 + acc1;
      for (int o = Lr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (sub == 0 && j < n_own) {
        const bool act = acc + ownpb[j] > a.tau;
        if (!lookahead) s_act[j] = act ? 1 : 0;
        if (act && sc_out != nullptr) {
          const int i = c + j * G;
          atomicOr(&sc_out[i >> 5], 1u << (i & 31));
        }
      }
    }
  } else {
    // Rows too many to stage: one warp per task reads each row from L2
    // (warmed in phase 0), lane l holding chunks l, l+32, ...; rows are
    // summed with a warp all-reduce and lane k keeps row k's score.  A task
    // is a whole 32-row word while a round of eight words is left, then a
    // quarter of a word: one warp per word left three warps working through
    // the last three words' round trips while five idled (the OPT-175B
    // shape: 11 words a block).
    float hreg[CPL][E];
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
      const int ch = lane + 32 * cc;
#pragma unroll
      for (int e = 0; e < E; ++e) hreg[cc][e] = ch < NC ? hs[ch * E + e] : 0.f;
    }
    const T* Ug = static_cast<const T*>(a.U);
    // rows in batches of UB, every load of a batch issued before any is used
    // (each row is an L2 round trip otherwise); wide forms have the registers
    constexpr int UB = CPT >= 4 ? 8 : 2;
    const int nfull = nwords / kLayerWarps * kLayerWarps;
    const int ntask = nfull + 4 * (nwords - nfull);
    for (int t = warp; t < ntask; t += kLayerWarps) {
      const int q = t < nfull ? t : nfull + (t - nfull) / 4;
      const int kb = t < nfull ? 0 : ((t - nfull) % 4) * 8;
      const int ke = t < nfull ? 32 : kb + 8;
      const int kn = min(ke, n_own - q * 32);
      float mine = 0.f;
      for (int k0 = kb; k0 < kn; k0 += UB) {
        uint4 raw[UB][CPL];
#pragma unroll
        for (int u = 0; u < UB; ++u)
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) {
            const int ch = lane + 32 * cc;
            const int j = q * 32 + k0 + u;
            raw[u][cc] = k0 + u < kn && ch < NC ? ldg_stream(Ug + (size_t)(c + (size_t)j * G) * r + ch * E)
                                                : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
          float acc = 0.f;
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) {
            float w[E];
            unpack<T>(raw[u][cc], w);
#pragma unroll
            for (int e = 0; e < E; ++e) acc = fmaf(w[e], hreg[cc][e], acc);
          }
          acc = warp_sum(acc);
          if (lane == k0 + u) mine = acc;
        }
      }
      const int j = q * 32 + lane;
      const bool mine_ok = lane >= kb && lane < kn;
      const bool act = mine_ok && (mine + ownpb[mine_ok ? j : 0]) > a.tau;
      if (mine_ok && !lookahead) s_act[j] = act ? 1 : 0;
      if (act && sc_out != nullptr) {
        const int i = c + j * G;
        atomicOr(&sc_out[i >> 5], 1u << (i & 31));
      }
    }
  }
  __syncthreads();
  SFFN_TRACE(9);
  if (ponly) {  // the predictor's mask words are out: nothing else to do
    cp_async_wait_all();
    return;
  }
  if (!lookahead) start_ring();
  // The pair split is settled when the ring first needs a list position it
  // may give away (k_safe and beyond): the rows below k_safe are this
  // block's whatever the partner sends, so the ring starts on them without
  // waiting for the partner's message, which has long arrived when the split
  // is settled.  Look-ahead calls settle here (their ring began earlier).
  bool settled = a.cluster != 2 || lookahead;
  if (lookahead && !settle_ring()) return;
  if (settled) SFFN_TRACE_VAL(19, nloc);


  // ---- balancing: each token's active rows fall unevenly on the blocks (a
  // sum of independent Bernoulli draws per block), and the block with the
  // most rows sets the kernel's length.  Every block publishes its count and
  // list; once it has seen every block's count of this launch, every block
  // computes the same assignment: the total N gives capacities K or K + 1, each block keeps its
  // own rows up to max(capacity, prefill) -- its hot rows stay local -- and
  // the rows above that, in block order, fill the other blocks' free
  // capacity in block order.
  if (a.balance) {
    // publish: the list as {neuron, bias} pairs, then the count tagged with
    // this launch's tag, released after the pairs
    int2* pub = reinterpret_cast<int2*>(a.bal_lists) + (size_t)c * own_cap;
    for (int p = tid; p < nloc; p += kLayerThreads) pub[p] = make_int2(list[p], __float_as_int(lbias[p]));
    __syncthreads();
    if (tid == kBarrierThread) {  // its warp has no copies in flight, so the fence is short
      __threadfence();
      const uint64_t word = ((uint64_t)tag << 32) | (uint32_t)nloc;
      asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a.bal_counts + c), "l"(word) : "memory");
      SFFN_TRACE_AT(15, kBarrierThread);
    }
    if (warp == 0) {
      // every block's count, all loads in flight together, re-polling
      // (bounded) only the ones not yet published
      constexpr int kCnt = 8;  // counts per lane: up to 256 blocks
      uint64_t v[kCnt];
#pragma unroll
      for (int k = 0; k < kCnt; ++k) {
        const int cc = lane + 32 * k;
        v[k] = 0;
        if (cc < G) asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v[k]) : "l"(a.bal_counts + cc) : "memory");
      }
      bool ok = true;
      const uint64_t t0 = globaltimer_ns();
      while (true) {
        bool all = true;
#pragma unroll
        for (int k = 0; k < kCnt; ++k) {
          const int cc = lane + 32 * k;
          if (cc < G && (uint32_t)(v[k] >> 32) != tag) {
            all = false;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v[k]) : "l"(a.bal_counts + cc) : "memory");
          }
        }
        if (all) break;
        if (globaltimer_ns() - t0 > a.wait_ns) {
          set_status(a.hdr, kStTimeout, 0x306u);
          ok = false;
          break;
        }
      }
      int N = 0;
#pragma unroll
      for (int k = 0; k < kCnt; ++k) {
        const int cc = lane + 32 * k;
        const int n = cc < G ? (int)(uint32_t)v[k] : 0;
        if (cc < G) bal_cnt[cc] = n;
        N += n;
      }
      N = __reduce_add_sync(0xffffffffu, N);
      __syncwarp();
      SFFN_TRACE(16);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        const int K = N / G, R = N - K * G;
        int run_e = 0, run_d = 0, my_d = 0, my_def = 0, my_keep = 0;
        for (int q0 = 0; q0 < G; q0 += 32) {
          const int cc = q0 + lane;
          const int n = cc < G ? bal_cnt[cc] : 0;
          const int cap = K + (cc < R ? 1 : 0);
          const int keep = min(n, max(cap, P));
          const int exc = cc < G ? n - keep : 0;
          const int def = cc < G ? max(0, cap - keep) : 0;
          int ie = exc, id = def;  // inclusive warp scans
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int ve = __shfl_up_sync(0xffffffffu, ie, o), vd = __shfl_up_sync(0xffffffffu, id, o);
            if (lane >= o) {
              ie += ve;
              id += vd;
            }
          }
          if (cc < G) {
            bal_keep[cc] = keep;
            bal_einc[cc] = run_e + ie;
          }
          if (cc == c) {
            my_d = run_d + id - def;
            my_def = def;
            my_keep = keep;
          }
          run_e += __shfl_sync(0xffffffffu, ie, 31);
          run_d += __shfl_sync(0xffffffffu, id, 31);
        }
        my_d = __reduce_add_sync(0xffffffffu, my_d);  // only the lane holding block c contributes
        my_def = __reduce_add_sync(0xffffffffu, my_def);
        my_keep = __reduce_add_sync(0xffffffffu, my_keep);
        __syncwarp();
        const int X = run_e;  // rows given away in total
        const int nsteal = max(0, min(my_d + my_def, X) - my_d);
        for (int t = lane; t < nsteal; t += 32) {
          const int x = my_d + t;
          int lo = 0, hi = G - 1;  // first block whose inclusive prefix exceeds x
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (bal_einc[mid] > x)
              hi = mid;
            else
              lo = mid + 1;
          }
          const int owner_exc = bal_cnt[lo] - bal_keep[lo];
          const int pos = bal_keep[lo] + (x - (bal_einc[lo] - owner_exc));
          const int2 e = __ldcg(reinterpret_cast<const int2*>(a.bal_lists) + (size_t)lo * own_cap + pos);
          list[my_keep + t] = e.x;
          lbias[my_keep + t] = __int_as_float(e.y);
        }
        if (lane == 0) s_nloc = my_keep + nsteal;
        SFFN_TRACE(17);
      }
      if (lane == 0) s_passed = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_passed) {
      cp_async_wait_all();
      return;
    }
    nloc = s_nloc;
    SFFN_TRACE(14);
    for (int p = pre; p < min(S, nloc); ++p) fill(p % S, list[p]);
  }

  bool failed = false;
  float xr[CPT][E], yacc[CPT][E];
#pragma unroll
  for (int cq = 0; cq < CPT; ++cq) {
    const int ch = tid + cq * kLayerThreads;
    unpack<T>(ch < NCH ? xpk[cq] : make_uint4(0, 0, 0, 0), xr[cq]);
#pragma unroll
    for (int e = 0; e < E; ++e) yacc[cq][e] = 0.f;
  }
  // Groups of up to kGroup list positions; st0 and ph0 are the stage and the
  // barrier phase of the group's first position (advanced, not divided out).
  const int ng_max = max(1, min(kGroup, S / 2));
  int grp = 0, st0 = 0;
  uint32_t ph0 = 0;
  for (int p0 = 0, ng = 0; !settled || p0 < nloc; p0 += ng, ++grp) {
    // this group's positions and refills stay below k_safe, or the split is
    // settled first (at the latest when p0 reaches k_safe)
    if (!settled && p0 + ng_max + S > k_safe) {
      if (!settle_ring()) return;
      settled = true;
      SFFN_TRACE_VAL(19, nloc);
      // the refills the ring deferred: positions [k_safe, p0 + S)
      for (int q = max(k_safe, S); q < min(p0 + S, nloc); ++q) fill(q % S, list[q]);
      if (p0 >= nloc) break;
    }
    // the first group is the prefetched hot rows alone, so it need not wait for a cold row
    ng = (grp == 0 && n_hot > 0) ? min(n_hot, ng_max) : min(ng_max, nloc - p0);
    bool ok = true;
    int stg[kGroup];
    float pu[kGroup], pg[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      pu[g] = pg[g] = 0.f;
      int st = st0 + g;
      uint32_t ph = ph0;
      if (st >= S) {
        st -= S;
        ph ^= 1u;
      }
      stg[g] = st;
      if (g < ng) {
        if (!mbar_try_wait(&bars[st], ph)) ok &= layer_wait_slow(&bars[st], ph, a.hdr, a.wait_ns);
        const uint4* up = reinterpret_cast<const uint4*>(region + (size_t)st * stage_bytes);
#pragma unroll
        for (int cq = 0; cq < CPT; ++cq) {
          const int ch = tid + cq * kLayerThreads;
          if (ch < NCH) {
            float w[E];
            unpack<T>(up[ch], w);
#pragma unroll
            for (int e = 0; e < E; ++e) pu[g] = fmaf(w[e], xr[cq][e], pu[g]);
            if (reglu) {
              unpack<T>(up[NCH + ch], w);
#pragma unroll
              for (int e = 0; e < E; ++e) pg[g] = fmaf(w[e], xr[cq][e], pg[g]);
            }
          }
        }
      }
    }
    if (grp == 0) SFFN_TRACE(10);
    SFFN_TRACE_GROUP(3 * grp);
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      pu[g] = warp_sum(pu[g]);
      if (reglu) pg[g] = warp_sum(pg[g]);
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        s_red[grp & 1][warp][g][0] = pu[g];
        if (reglu) s_red[grp & 1][warp][g][1] = pg[g];
      }
    }
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    SFFN_TRACE_GROUP(3 * grp + 1);
    float act[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      float u = 0.f, gt = 0.f;
#pragma unroll
      for (int w = 0; w < kLayerWarps; ++w) {
        u += s_red[grp & 1][w][g][0];
        if (reglu) gt += s_red[grp & 1][w][g][1];
      }
      const float bias = g < ng ? lbias[p0 + g] : -INFINITY;
      act[g] = bias == -INFINITY ? 0.f : (reglu ? fmaxf(gt + bias, 0.f) * u : fmaxf(u + bias, 0.f));
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      if (g < ng) {
        const int st = stg[g];
        if (act[g] != 0.f) {
          const uint4* dn = reinterpret_cast<const uint4*>(region + (size_t)st * stage_bytes) + (size_t)(nrows - 1) * NCH;
#pragma unroll
          for (int cq = 0; cq < CPT; ++cq) {
            const int ch = tid + cq * kLayerThreads;
            if (ch < NCH) {
              float w[E];
              unpack<T>(dn[ch], w);
#pragma unroll
              for (int e = 0; e < E; ++e) yacc[cq][e] = fmaf(act[g], w[e], yacc[cq][e]);
            }
          }
        }
        // this thread is done with its chunks of the stage: refill them
        // (position p0 + g + S maps to the same stage; before the split is
        // settled, only positions below k_safe)
        if (p0 + g + S < (settled ? nloc : k_safe)) fill(st, list[p0 + g + S]);
      }
    }
    st0 += ng;
    if (st0 >= S) {
      st0 -= S;
      ph0 ^= 1u;
    }
    SFFN_TRACE_GROUP(3 * grp + 2);
  }
  if (failed) {
    cp_async_wait_all();
    if (a.cluster == 2) {  // phase 2 of the pair exchange (arrived here if the split was not settled)
      if (!settled) cluster_arrive();
      cluster_wait();
    }
    return;
  }

  // ---- phase 6: add this block's contribution into y
  SFFN_TRACE(6);
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
  SFFN_TRACE(7);
  if (a.cluster == 2) cluster_wait();  // phase 2 of the pair exchange
}


// The dynamic shared-memory limit set so far for k_layer<T, CPT, ACT> (raised, never lowered).
template <typename T, int CPT, int ACT>
int& layer_smem_limit() {
  static int cur = 48 * 1024;
  return cur;
}

// k_layer for the configuration's activation, with its shared-memory limit raised to cfg.smem.
template <typename T, int CPT>
void (*layer_kernel(const LayerConfig& cfg, cudaError_t* err))(LayerArgs) {
  if (cfg.act == kReglu) {
    *err = ensure_dyn_smem(k_layer<T, CPT, kReglu>, cfg.smem, &layer_smem_limit<T, CPT, kReglu>());
    return k_layer<T, CPT, kReglu>;
  }
  *err = ensure_dyn_smem(k_layer<T, CPT, kRelu>, cfg.smem, &layer_smem_limit<T, CPT, kRelu>());
  return k_layer<T, CPT, kRelu>;
}

template <typename T, int CPT>
cudaError_t layer_launch(const LayerConfig& cfg, const LayerArgs& a, int grid, cudaStream_t s) {
  if (a.act != cfg.act) return cudaErrorInvalidValue;
  cudaError_t e;
  void (*kern)(LayerArgs) = layer_kernel<T, CPT>(cfg, &e);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: this kernel may start while the previous
  // kernel on the stream finishes; it waits for it (griddepcontrol.wait)
  // before touching anything that kernel may write.
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kLayerThreads);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.cluster > 1 ? a.cluster : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = a.cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&lc, kern, a);
}

template <typename T, int CPT>
int layer_occupancy(const LayerConfig& cfg) {
  cudaError_t e;
  void (*kern)(LayerArgs) = layer_kernel<T, CPT>(cfg, &e);
  if (e != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kLayerThreads, cfg.smem) != cudaSuccess) return 0;
  return n;
}

template <typename T, int CPT>
int layer_clusters(const LayerConfig& cfg, int grid, int cs) {
  cudaError_t e;
  void (*kern)(LayerArgs) = layer_kernel<T, CPT>(cfg, &e);
  if (e != cudaSuccess) return 0;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kLayerThreads);
  lc.dynamicSmemBytes = cfg.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess) return 0;
  return n;
}

template <typename T>
int layer_max_clusters_t(const LayerConfig& cfg, int grid, int cs) {
  switch (cfg.cpt) {
    case 1: return layer_clusters<T, 1>(cfg, grid, cs);
    case 2: return layer_clusters<T, 2>(cfg, grid, cs);
    case 3: return layer_clusters<T, 3>(cfg, grid, cs);
    case 4: return layer_clusters<T, 4>(cfg, grid, cs);
    case 6: return layer_clusters<T, 6>(cfg, grid, cs);
  }
  return 0;
}

template <typename T>
int layer_blocks_per_sm_t(const LayerConfig& cfg) {
  switch (cfg.cpt) {
    case 1: return layer_occupancy<T, 1>(cfg);
    case 2: return layer_occupancy<T, 2>(cfg);
    case 3: return layer_occupancy<T, 3>(cfg);
    case 4: return layer_occupancy<T, 4>(cfg);
    case 6: return layer_occupancy<T, 6>(cfg);
  }
  return 0;
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
