// Online activation predictor: h = V x, s = U h + pb, mask = s > tau, and the
// compaction of the mask into ascending neuron-index lists.
//
// The pages describe the predictor only in prose (PowerInfer page,
// "Predictores de espacialidad adaptativa": a small per-layer predictor kept on
// the GPU scores the neurons and only those predicted active are computed).
// Here it is the rank-r linear scorer; both GEMVs are HBM-bound reads of V and
// U and are laid out for full-width 16-byte coalesced loads.

#include "kernels.cuh"

namespace sffn {

namespace {

constexpr int kHiddenWarps = 8;
// Rows of V per warp: two for up to 8 tokens per block, one beyond (the
// 2 x BT accumulators would otherwise limit a 32-token block to one per SM).
template <int BT> struct HiddenRows {
  static constexpr int kPerWarp = BT <= 8 ? 2 : 1;
  static constexpr int kPerBlock = kHiddenWarps * kPerWarp;
};
constexpr int kHiddenRowsPerBlockMin = kHiddenWarps;  // the smallest row group (most groups)

// Grid (KS, row groups, token groups).  Each block stages its K-chunk of the
// BT tokens in shared memory; each warp streams two rows of V over the chunk.
// Partial sums go to h_part; the last block of a (row group, token group) to
// arrive sums the KS partials in a fixed order, so h is deterministic.
template <typename T, int BT>
__global__ void __launch_bounds__(kHiddenWarps * 32)
    k_pred_hidden(const T* __restrict__ V, const T* __restrict__ x, int B, int r, int d, int kc_elems,
                  int KS, float* __restrict__ h_part, float* __restrict__ h, uint32_t* __restrict__ tickets,
                  T* __restrict__ h3) {
  constexpr int E = Chunk<T>::N;
  extern __shared__ uint4 xs[];  // [BT][kc_elems / E]
  __shared__ uint32_t s_last;
  const int ks = blockIdx.x, rg = blockIdx.y, tg = blockIdx.z;
  const int b0 = tg * BT;
  const int k0 = ks * kc_elems;
  const int nch = min(kc_elems, d - k0) / E;
  const int cstride = kc_elems / E;

  for (int i = threadIdx.x; i < BT * nch; i += blockDim.x) {
    const int bb = i / nch, c = i - bb * nch;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (b0 + bb < B) v = *reinterpret_cast<const uint4*>(x + (size_t)(b0 + bb) * d + k0 + c * E);
    xs[bb * cstride + c] = v;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kHiddenRowsPerWarp = HiddenRows<BT>::kPerWarp;
  constexpr int kHiddenRowsPerBlock = HiddenRows<BT>::kPerBlock;
  const int row0 = rg * kHiddenRowsPerBlock + warp * kHiddenRowsPerWarp;
  float acc[kHiddenRowsPerWarp][BT];
#pragma unroll
  for (int q = 0; q < kHiddenRowsPerWarp; ++q)
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) acc[q][bb] = 0.f;

#pragma unroll 4
  for (int c = lane; c < nch; c += 32) {
    uint4 raw[kHiddenRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kHiddenRowsPerWarp; ++q) {
      const int row = row0 + q;
      raw[q] = row < r ? ldg_stream(V + (size_t)row * d + k0 + c * E) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) {
      float xv[E];
      unpack<T>(xs[bb * cstride + c], xv);
#pragma unroll
      for (int q = 0; q < kHiddenRowsPerWarp; ++q) {
        float w[E];
        unpack<T>(raw[q], w);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[q][bb] = fmaf(w[e], xv[e], acc[q][bb]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kHiddenRowsPerWarp; ++q) {
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) {
      const float v = warp_sum(acc[q][bb]);
      const int row = row0 + q;
      if (lane == 0 && row < r && b0 + bb < B) h_part[((size_t)ks * B + b0 + bb) * r + row] = v;
    }
  }

  // Last arriving K-chunk block of this (row group, token group) reduces.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    uint32_t* t = &tickets[rg * gridDim.z + tg];
    const uint32_t prev = atomicAdd(t, 1u);
    s_last = (prev == (uint32_t)KS - 1u);
    if (s_last) {
      atomicExch(t, 0u);
      __threadfence();
    }
  }
  __syncthreads();
  if (!s_last) return;
  for (int i = threadIdx.x; i < kHiddenRowsPerBlock * BT; i += blockDim.x) {
    const int q = i / BT, bb = i - q * BT;
    const int row = rg * kHiddenRowsPerBlock + q;
    if (row >= r || b0 + bb >= B) continue;
    // fixed summation order; eight partial-sum loads in flight at a time
    float s = 0.f;
    const float* hp = h_part + (size_t)(b0 + bb) * r + row;
    const size_t kstride = (size_t)B * r;
    int k = 0;
    for (; k + 8 <= KS; k += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(hp + (size_t)(k + u) * kstride);
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; k < KS; ++k) s += __ldcg(hp + (size_t)k * kstride);
    h[(size_t)(b0 + bb) * r + row] = s;
    if (h3 != nullptr) {  // three 16-bit parts whose sum carries the fp32 value
      const T hi = from_float<T>(s);
      const float rest = s - static_cast<float>(hi);
      const T mid = from_float<T>(rest);
      const T lo = from_float<T>(rest - static_cast<float>(mid));
      h3[(size_t)(0 * BT + bb) * r + row] = hi;
      h3[(size_t)(1 * BT + bb) * r + row] = mid;
      h3[(size_t)(2 * BT + bb) * r + row] = lo;
    }
  }
}

// Hidden layer for a batch of up to 32 tokens, lane = token.  Grid (KS row
// K-chunks, r / 32 row groups).  A block stages its 32 rows of V and the
// tokens' K-chunk in shared memory as fp32 (token rows padded so the lanes'
// float4 loads spread over the banks); warp w accumulates rows 4w .. 4w+3
// for token `lane` over the chunk -- no cross-lane reduction -- and writes
// the partial sums; the last block of a row group to arrive sums the KS
// partials in a fixed order, writes h and, for the tensor-core score
// product, h as three 16-bit parts.
constexpr int kTokRows = 32;   // rows of V per block
constexpr int kTokKc = 256;    // K-chunk

template <typename T>
__global__ void __launch_bounds__(256)
    k_pred_hidden_tok(const T* __restrict__ V, const T* __restrict__ x, int B, int r, int d, int KS,
                      float* __restrict__ h_part, float* __restrict__ h, uint32_t* __restrict__ tickets,
                      T* __restrict__ h3, int BT) {
  constexpr int E = Chunk<T>::N;
  constexpr int XP = kTokKc + 4;  // padded token row (floats)
  extern __shared__ __align__(16) float tok_smem[];
  float(*vs)[kTokKc] = reinterpret_cast<float(*)[kTokKc]>(tok_smem);                 // [kTokRows][kTokKc]
  float(*xs)[XP] = reinterpret_cast<float(*)[XP]>(tok_smem + kTokRows * kTokKc);     // [32][XP]
  __shared__ uint32_t s_last;
  const int ks = blockIdx.x, rg = blockIdx.y;
  const int k0 = ks * kTokKc, kn = min(kTokKc, d - k0);
  const int row0 = rg * kTokRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nchk = kn / E;  // 16-byte chunks of the K-chunk per row
  for (int i = tid; i < kTokRows * nchk; i += 256) {
    const int rr = i / nchk, c = i - rr * nchk;
    float v[E];
    if (row0 + rr < r)
      unpack<T>(ldg_stream(V + (size_t)(row0 + rr) * d + k0 + c * E), v);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) vs[rr][c * E + e] = v[e];
  }
  for (int i = tid; i < 32 * nchk; i += 256) {
    const int bb = i / nchk, c = i - bb * nchk;
    float v[E];
    if (bb < B)
      unpack<T>(*reinterpret_cast<const uint4*>(x + (size_t)bb * d + k0 + c * E), v);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) xs[bb][c * E + e] = v[e];
  }
  __syncthreads();
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const float* xr = xs[lane];
#pragma unroll 4
  for (int k = 0; k < kn; k += 4) {
    const float4 xv = *reinterpret_cast<const float4*>(xr + k);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 vv = *reinterpret_cast<const float4*>(&vs[warp * 4 + q][k]);
      acc[q] = fmaf(vv.x, xv.x, fmaf(vv.y, xv.y, fmaf(vv.z, xv.z, fmaf(vv.w, xv.w, acc[q]))));
    }
  }
  const int rowq = row0 + warp * 4;
  if (lane < B) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (rowq + q < r) h_part[((size_t)ks * B + lane) * r + rowq + q] = acc[q];
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    uint32_t* t = &tickets[rg];
    const uint32_t prev = atomicAdd(t, 1u);
    s_last = (prev == (uint32_t)KS - 1u);
    if (s_last) {
      atomicExch(t, 0u);
      __threadfence();
    }
  }
  __syncthreads();
  if (!s_last) return;
  for (int i = tid; i < kTokRows * B; i += 256) {
    const int bb = i / kTokRows, q = i - bb * kTokRows;
    const int row = row0 + q;
    if (row >= r) continue;
    const float* hp = h_part + (size_t)bb * r + row;
    const size_t kstride = (size_t)B * r;
    float sum = 0.f;
    int k = 0;
    for (; k + 8 <= KS; k += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(hp + (size_t)(k + u) * kstride);
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += v[u];
    }
    for (; k < KS; ++k) sum += __ldcg(hp + (size_t)k * kstride);
    h[(size_t)bb * r + row] = sum;
    if (h3 != nullptr) {  // three 16-bit parts whose sum carries the fp32 value
      const T hi = from_float<T>(sum);
      const float rest = sum - static_cast<float>(hi);
      const T mid = from_float<T>(rest);
      const T lo = from_float<T>(rest - static_cast<float>(mid));
      h3[(size_t)(0 * BT + bb) * r + row] = hi;
      h3[(size_t)(1 * BT + bb) * r + row] = mid;
      h3[(size_t)(2 * BT + bb) * r + row] = lo;
    }
  }
}

// Hidden layer for a batch of 8 to 32 tokens, 16-bit weights, feeding the
// tensor-core score product (h also as three 16-bit parts).  Clusters of
// eight blocks: cluster y owns rows [16y, 16y + 16) of V and block q of it the
// q-th eighth of d.  A block copies its V rows and the tokens' columns into
// shared memory with cp.async in four groups along d, and works on each group
// as soon as it has landed, so the copies of the later groups overlap the
// arithmetic of the earlier ones.  Every lane owns a micro-tile of 4 rows x 4
// tokens and a share of the 16-byte column pieces (the lanes of a warp that
// hold the same micro-tile take neighbouring pieces and are summed by
// shuffles at the end); pieces are stored at permuted positions so that the
// distinct addresses of one warp-wide load fall in distinct banks as far as
// their number allows.  The warps' partial sums are added in shared memory,
// and after a cluster barrier block q sums rows 2q, 2q + 1 of the cluster's
// tile over the eight blocks' shared memory.  Every sum runs in a fixed
// order, so h is the same from run to run; there are no global partial sums
// and no arrival counters.
constexpr int kHcCL = 8;         // blocks per cluster: the split of d
constexpr int kHcRows = 16;      // rows of V per cluster
constexpr int kHcThreads = 256;  // eight warps
constexpr int kHcPieces = 12;    // 16-byte loads in flight per thread

__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int BT> struct HcTile {
  static constexpr int MR = 4, MB = 4;       // micro-tile: rows x tokens per lane
  static constexpr int NRG = kHcRows / MR;   // row groups (4)
  static constexpr int NTG = BT / MB;        // token groups (2, 4, 8)
  static constexpr int LPC = NRG * NTG;      // lanes per column piece
  static constexpr int KQ = 32 / LPC;        // lanes holding the same micro-tile (4, 2, 1)
  static_assert(LPC * KQ == 32, "whole warps");
};

// Piece positions: V row rr, piece c at c ^ vperm(rr); token b at c ^ xperm(b).
__device__ __forceinline__ int hc_vperm(int rr) { return (rr >> 1) & 6; }
template <int BT> __device__ __forceinline__ int hc_xperm(int b) { return ((b >> 2) * HcTile<BT>::KQ) & 7; }

template <int BT>
size_t hidden_cl_smem(int d) {
  const size_t nchk = (size_t)d / kHcCL / 8;
  return (kHcRows + BT) * nchk * 16 + (size_t)(kHcThreads / 32 + 1) * kHcRows * BT * 4;
}

template <typename T, int BT>
__global__ void __cluster_dims__(kHcCL, 1, 1) __launch_bounds__(kHcThreads)
    k_pred_hidden_cl(const T* __restrict__ V, const T* __restrict__ x, int B, int r, int d,
                     float* __restrict__ h, T* __restrict__ h3) {
  using Tile = HcTile<BT>;
  constexpr int MR = Tile::MR, MB = Tile::MB, NTG = Tile::NTG, LPC = Tile::LPC, KQ = Tile::KQ;
  constexpr int kWarps = kHcThreads / 32;
  extern __shared__ __align__(16) unsigned char hc_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = (int)cluster_rank();
  const int row0 = blockIdx.y * kHcRows;
  const int Kc = d / kHcCL;   // a multiple of 64
  const int nchk = Kc / 8;    // 16-byte pieces of a row's part (a multiple of 8)
  const int k0 = q * Kc;
  uint4* vs = reinterpret_cast<uint4*>(hc_smem);           // [kHcRows][nchk]
  uint4* xs = vs + kHcRows * nchk;                          // [BT][nchk]
  float* part = reinterpret_cast<float*>(xs + BT * nchk);  // [warp][row][token]
  float* P = part + kWarps * kHcRows * BT;                 // [row][token], this block's part of d

  // copies: every piece through registers (16-byte loads, up to kHcPieces
  // in flight per thread per round), then into its permuted position
  const int npieces = (kHcRows + BT) * nchk;
  for (int p0 = 0; p0 < npieces; p0 += kHcPieces * kHcThreads) {
    uint4 reg[kHcPieces];
#pragma unroll
    for (int u = 0; u < kHcPieces; ++u) {
      const int i = p0 + u * kHcThreads + tid;
      const int rowi = i / nchk, c = i - rowi * nchk;
      reg[u] = make_uint4(0, 0, 0, 0);
      if (i < npieces) {
        if (rowi < kHcRows) {
          if (row0 + rowi < r) reg[u] = ldg_stream(V + (size_t)(row0 + rowi) * d + k0 + c * 8);
        } else if (rowi - kHcRows < B) {
          reg[u] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(rowi - kHcRows) * d + k0 + c * 8));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kHcPieces; ++u) {
      const int i = p0 + u * kHcThreads + tid;
      const int rowi = i / nchk, c = i - rowi * nchk;
      if (i < npieces) {
        if (rowi < kHcRows)
          vs[rowi * nchk + (c ^ hc_vperm(rowi))] = reg[u];
        else
          xs[(rowi - kHcRows) * nchk + (c ^ hc_xperm<BT>(rowi - kHcRows))] = reg[u];
      }
    }
  }
  __syncthreads();

  const int kq = lane / LPC, within = lane - kq * LPC;
  const int rg = within / NTG, tg = within - rg * NTG;
  const int vp = hc_vperm(rg * MR), xp = hc_xperm<BT>(tg * MB);
  float acc[MR][MB];
#pragma unroll
  for (int i = 0; i < MR; ++i)
#pragma unroll
    for (int j = 0; j < MB; ++j) acc[i][j] = 0.f;
  for (int c = warp * KQ + kq; c < nchk; c += kWarps * KQ) {
    float w[MR][8], xv[MB][8];
#pragma unroll
    for (int i = 0; i < MR; ++i) unpack<T>(vs[(rg * MR + i) * nchk + (c ^ vp)], w[i]);
#pragma unroll
    for (int j = 0; j < MB; ++j) unpack<T>(xs[(tg * MB + j) * nchk + (c ^ xp)], xv[j]);
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int j = 0; j < MB; ++j) acc[i][j] = fmaf(w[i][e], xv[j][e], acc[i][j]);
  }

  // the lanes holding the same micro-tile, then the warps, in a fixed order
#pragma unroll
  for (int i = 0; i < MR; ++i)
#pragma unroll
    for (int j = 0; j < MB; ++j)
#pragma unroll
      for (int o = LPC; o < 32; o <<= 1) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], o);
  if (kq == 0)
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
      for (int j = 0; j < MB; ++j) part[(warp * kHcRows + rg * MR + i) * BT + tg * MB + j] = acc[i][j];
  __syncthreads();
  for (int o = tid; o < kHcRows * BT; o += kHcThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sum += part[w * kHcRows * BT + o];
    P[o] = sum;
  }
  cluster_arrive();  // release: this block's P is complete
  cluster_wait();    // acquire: every block's P is complete

  constexpr int kRowsPerBlock = kHcRows / kHcCL;
  if (tid < kRowsPerBlock * BT) {
    const int rr = q * kRowsPerBlock + tid / BT, b = tid % BT;
    float v[kHcCL];
#pragma unroll
    for (int p = 0; p < kHcCL; ++p) v[p] = ld_peer_f32(peer_smem(P + rr * BT + b, (uint32_t)p));
    float sum = 0.f;
#pragma unroll
    for (int p = 0; p < kHcCL; ++p) sum += v[p];
    const int row = row0 + rr;
    if (row < r && b < B) {
      h[(size_t)b * r + row] = sum;
      // three 16-bit parts whose sum carries the fp32 value
      const T hi = from_float<T>(sum);
      const float rest = sum - static_cast<float>(hi);
      const T mid = from_float<T>(rest);
      const T lo = from_float<T>(rest - static_cast<float>(mid));
      h3[(size_t)(0 * BT + b) * r + row] = hi;
      h3[(size_t)(1 * BT + b) * r + row] = mid;
      h3[(size_t)(2 * BT + b) * r + row] = lo;
    }
  }
  cluster_arrive();  // no block leaves while another may still read its P
  cluster_wait();
}

// Scores.  A block owns 64-row blocks (two mask words) in a grid-stride loop;
// each warp streams 8 rows of U, lane l holding the 16-byte chunks l, l+32, ...
// of every row (CPL chunks), and rows are summed with a warp all-reduce.
constexpr int kScoreWarps = 8;
constexpr int kScoreRowsPerWarp = 8;
constexpr int kScoreRowsPerBlock = kScoreWarps * kScoreRowsPerWarp;  // 64 = 2 words

template <typename T, int CPL, int BT>
__global__ void __launch_bounds__(kScoreWarps * 32)
    k_pred_score(const T* __restrict__ U, const float* __restrict__ h, const float* __restrict__ pb,
                 float tau, int B, int f, int r, int W, uint32_t* __restrict__ mask,
                 float* __restrict__ scores) {
  constexpr int E = Chunk<T>::N;
  constexpr int RIF = (8 / CPL) > 0 ? (8 / CPL) : 1;  // rows in flight per warp
  extern __shared__ float hs[];                        // [BT][r]
  __shared__ uint32_t s_words[BT][2];
  const int b0 = blockIdx.y * BT;
  const int nb = min(BT, B - b0);
  const int NC = r / E;  // chunks per row

  for (int i = threadIdx.x; i < BT * r; i += blockDim.x) {
    const int bb = i / r;
    hs[i] = bb < nb ? h[(size_t)(b0 + bb) * r + (i - bb * r)] : 0.f;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int blk = blockIdx.x; blk * kScoreRowsPerBlock < f; blk += gridDim.x) {
    if (threadIdx.x < 2 * BT) s_words[threadIdx.x >> 1][threadIdx.x & 1] = 0u;
    __syncthreads();
    const int wrow0 = blk * kScoreRowsPerBlock + warp * kScoreRowsPerWarp;
    uint32_t bits[BT];
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) bits[bb] = 0u;

#pragma unroll
    for (int g = 0; g < kScoreRowsPerWarp; g += RIF) {
      uint4 raw[RIF][CPL];
#pragma unroll
      for (int q = 0; q < RIF; ++q) {
        const int row = wrow0 + g + q;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane + 32 * c;
          raw[q][c] = (row < f && ch < NC) ? ldg_stream(U + (size_t)row * r + ch * E)
                                           : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int q = 0; q < RIF; ++q) {
        const int row = wrow0 + g + q;
        float acc[BT];
#pragma unroll
        for (int bb = 0; bb < BT; ++bb) acc[bb] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane + 32 * c;
          if (ch < NC) {
            float w[E];
            unpack<T>(raw[q][c], w);
#pragma unroll
            for (int bb = 0; bb < BT; ++bb) {
              const float* hp = hs + bb * r + ch * E;
#pragma unroll
              for (int e = 0; e < E; ++e) acc[bb] = fmaf(w[e], hp[e], acc[bb]);
            }
          }
        }
        const float bias = row < f ? __ldg(&pb[row]) : 0.f;
#pragma unroll
        for (int bb = 0; bb < BT; ++bb) {
          const float s = warp_sum(acc[bb]) + bias;
          if (row < f && s > tau) bits[bb] |= 1u << (g + q);
          if (scores != nullptr && lane == q && row < f && bb < nb) scores[(size_t)(b0 + bb) * f + row] = s;
        }
      }
    }
    if (lane == 0) {
      const int word_in_blk = warp >> 2, shift = (warp & 3) * kScoreRowsPerWarp;
#pragma unroll
      for (int bb = 0; bb < BT; ++bb) atomicOr(&s_words[bb][word_in_blk], bits[bb] << shift);
    }
    __syncthreads();
    if (threadIdx.x < 2 * BT) {
      const int bb = threadIdx.x >> 1, wi = threadIdx.x & 1;
      const int word = blk * 2 + wi;
      if (bb < nb && word < W) mask[(size_t)(b0 + bb) * W + word] = s_words[bb][wi];
    }
  }
}

// One block per token: exclusive scan of the popcounts of the mask words,
// then every set bit is written at its rank.
constexpr int kCompactThreads = 512;

__global__ void __launch_bounds__(kCompactThreads)
    k_compact(const uint32_t* __restrict__ mask, int f, int W, int32_t* __restrict__ idx,
              int32_t* __restrict__ n_active) {
  __shared__ int s_warp[kCompactThreads / 32];
  const int b = blockIdx.x;
  const uint32_t* m = mask + (size_t)b * W;
  const int wpt = (W + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * wpt;
  int cnt = 0;
  for (int k = 0; k < wpt; ++k)
    if (w0 + k < W) cnt += __popc(m[w0 + k]);
  // block exclusive scan of cnt
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < nw) s_warp[lane] = v;  // inclusive warp totals
  }
  __syncthreads();
  int pos = incl - cnt + (warp > 0 ? s_warp[warp - 1] : 0);
  int32_t* out = idx + (size_t)b * f;
  for (int k = 0; k < wpt; ++k) {
    const int w = w0 + k;
    if (w >= W) break;
    uint32_t bitsw = m[w];
    while (bitsw) {
      const int j = __ffs(bitsw) - 1;
      bitsw &= bitsw - 1;
      out[pos++] = w * 32 + j;
    }
  }
  if (threadIdx.x == blockDim.x - 1) n_active[b] = pos;
}

__global__ void k_count_bits(const uint32_t* __restrict__ mask, int B, int f, int W,
                             int32_t* __restrict__ counts) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < f; i += gridDim.x * blockDim.x) {
    int c = 0;
    for (int b = 0; b < B; ++b) c += (mask[(size_t)b * W + (i >> 5)] >> (i & 31)) & 1u;
    counts[i] += c;
  }
}

template <typename T, int BT>
cudaError_t hidden_launch(const PredHiddenArgs& a, cudaStream_t s) {
  const dim3 grid(a.KS, (a.r + HiddenRows<BT>::kPerBlock - 1) / HiddenRows<BT>::kPerBlock, (a.B + BT - 1) / BT);
  const size_t smem = (size_t)BT * a.kc_elems * sizeof(T);
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_pred_hidden<T, BT>, smem, &cur);
  if (e != cudaSuccess) return e;
  k_pred_hidden<T, BT><<<grid, kHiddenWarps * 32, smem, s>>>(
      static_cast<const T*>(a.V), static_cast<const T*>(a.x), a.B, a.r, a.d, a.kc_elems, a.KS,
      a.h_part, a.h, a.tickets, static_cast<T*>(a.h3));
  return cudaGetLastError();
}

template <typename T, int BT>
cudaError_t hidden_cl_launch(const PredHiddenArgs& a, cudaStream_t s) {
  const size_t smem = hidden_cl_smem<BT>(a.d);
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_pred_hidden_cl<T, BT>, smem, &cur);
  if (e != cudaSuccess) return e;
  const dim3 grid(kHcCL, (a.r + kHcRows - 1) / kHcRows);
  k_pred_hidden_cl<T, BT><<<grid, kHcThreads, smem, s>>>(static_cast<const T*>(a.V), static_cast<const T*>(a.x),
                                                          a.B, a.r, a.d, a.h, static_cast<T*>(a.h3));
  return cudaGetLastError();
}

template <typename T>
cudaError_t hidden_cl_dispatch(const PredHiddenArgs& a, cudaStream_t s) {
  switch (a.bt) {
    case 8: return hidden_cl_launch<T, 8>(a, s);
    case 16: return hidden_cl_launch<T, 16>(a, s);
    case 32: return hidden_cl_launch<T, 32>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t hidden_dispatch(const PredHiddenArgs& a, cudaStream_t s) {
  if (a.cluster) {
    if constexpr (sizeof(T) == 2) {
      if (a.h3 == nullptr || a.B > a.bt || a.d % (kHcCL * 64) != 0) return cudaErrorInvalidValue;
      return hidden_cl_dispatch<T>(a, s);
    } else {
      return cudaErrorInvalidValue;
    }
  }
  if (a.bt == 32 && a.B > 16) {  // one group of 17-32 tokens: lane = token kernel, K-chunks of 256
    if (a.B > 32 || a.kc_elems != kTokKc) return cudaErrorInvalidValue;
    const dim3 grid(a.KS, (a.r + kTokRows - 1) / kTokRows);
    const size_t smem = (size_t)(kTokRows * kTokKc + 32 * (kTokKc + 4)) * sizeof(float);
    static int cur = 48 * 1024;
    const cudaError_t e = ensure_dyn_smem(k_pred_hidden_tok<T>, smem, &cur);
    if (e != cudaSuccess) return e;
    k_pred_hidden_tok<T><<<grid, 256, smem, s>>>(static_cast<const T*>(a.V), static_cast<const T*>(a.x), a.B, a.r,
                                                 a.d, a.KS, a.h_part, a.h, a.tickets, static_cast<T*>(a.h3), a.bt);
    return cudaGetLastError();
  }
  if (a.bt == 8) return hidden_launch<T, 8>(a, s);
  if (a.bt == 16) return hidden_launch<T, 16>(a, s);
  if (a.bt == 32) return hidden_launch<T, 32>(a, s);
  if (a.bt != 0 || a.h3 != nullptr) return cudaErrorInvalidValue;
  if (a.B == 1) return hidden_launch<T, 1>(a, s);
  if (a.B == 2) return hidden_launch<T, 2>(a, s);
  if (a.B <= 4) return hidden_launch<T, 4>(a, s);
  return hidden_launch<T, 8>(a, s);
}

template <typename T, int CPL, int BT>
cudaError_t score_launch(const PredScoreArgs& a, cudaStream_t s) {
  const dim3 grid(a.grid, (a.B + BT - 1) / BT);
  const size_t smem = (size_t)BT * a.r * sizeof(float);
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_pred_score<T, CPL, BT>, smem, &cur);
  if (e != cudaSuccess) return e;
  k_pred_score<T, CPL, BT><<<grid, kScoreWarps * 32, smem, s>>>(
      static_cast<const T*>(a.U), a.h, a.pb, a.tau, a.B, a.f, a.r, a.W, a.mask, a.scores);
  return cudaGetLastError();
}

template <typename T, int CPL>
cudaError_t score_bt(const PredScoreArgs& a, cudaStream_t s) {
  if (a.B == 1) return score_launch<T, CPL, 1>(a, s);
  if (a.B == 2) return score_launch<T, CPL, 2>(a, s);
  if (a.B <= 4) return score_launch<T, CPL, 4>(a, s);
  return score_launch<T, CPL, 8>(a, s);
}

template <typename T>
cudaError_t score_dispatch(const PredScoreArgs& a, cudaStream_t s) {
  const int nc = a.r / Chunk<T>::N;
  if (nc <= 32) return score_bt<T, 1>(a, s);
  if (nc <= 64) return score_bt<T, 2>(a, s);
  if (nc <= 128) return score_bt<T, 4>(a, s);
  if (nc <= 256) return score_bt<T, 8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

// Row groups of the hidden-layer kernel at its smallest group size: an upper
// bound on the arrival tickets any launch uses per token group.
int pred_hidden_row_groups(int r) { return (r + kHiddenRowsPerBlockMin - 1) / kHiddenRowsPerBlockMin; }

size_t pred_hidden_cluster_smem(int d, int bt) {
  if (d % (kHcCL * 64) != 0) return 0;
  switch (bt) {
    case 8: return hidden_cl_smem<8>(d);
    case 16: return hidden_cl_smem<16>(d);
    case 32: return hidden_cl_smem<32>(d);
  }
  return 0;
}

cudaError_t launch_pred_hidden(int dtype, const PredHiddenArgs& a, cudaStream_t s) {
  switch (dtype) {
    case kF32: return hidden_dispatch<float>(a, s);
    case kF16: return hidden_dispatch<__half>(a, s);
    case kBF16: return hidden_dispatch<__nv_bfloat16>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_pred_score(int dtype, const PredScoreArgs& a, cudaStream_t s) {
  switch (dtype) {
    case kF32: return score_dispatch<float>(a, s);
    case kF16: return score_dispatch<__half>(a, s);
    case kBF16: return score_dispatch<__nv_bfloat16>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_compact(const uint32_t* mask, int B, int f, int W, int32_t* idx, int32_t* n_active,
                           cudaStream_t s) {
  k_compact<<<B, kCompactThreads, 0, s>>>(mask, f, W, idx, n_active);
  return cudaGetLastError();
}

cudaError_t launch_count_bits(const uint32_t* mask, int B, int f, int W, int32_t* counts, cudaStream_t s) {
  const int threads = 256;
  const int grid = (f + threads - 1) / threads;
  k_count_bits<<<grid, threads, 0, s>>>(mask, B, f, W, counts);
  return cudaGetLastError();
}

}  // namespace sffn
