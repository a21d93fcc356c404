// Predictor scores and threshold for a batch of 8 to 32 tokens on the tensor
// cores: s_i = U_i . h_b + pb_i, active <=> s_i > tau, written as mask words.
//
// The online predictor of the PowerInfer page ("Predictores de espacialidad
// adaptativa") scores every neuron of the layer for every token; for a batch
// that is the product S = U H, M = d_ff rows of U, K = rank, N = tokens.  The
// hidden vectors h (fp32, from the V x kernel) enter the MMA as three 16-bit
// parts, h = hi + mid + lo, stacked along N, so that the sum of the three
// products carries the fp32 value of h and the threshold is decided as it
// would be in fp32.
//
// Work: a block owns a contiguous range of mask words (32 neurons each) and
// walks it in tiles of up to 128 rows; per tile, jobs of 64 columns of the
// rank copy the tile's U rows and the three parts of every token into a slot
// of a cp.async ring (128-byte swizzled K-major tiles); one thread issues the
// MMAs into one of two tensor-memory accumulators; the epilogue warps add the
// parts and the bias, threshold, and ballot each warp's 32 rows into one mask
// word per token.

#pragma once

#include "kernels.cuh"
#include "tcgen05.cuh"

namespace sffn {
namespace sc {

using namespace tc;

constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarps = 8;
constexpr int kThreads = kScoreMmaThreads;
static_assert(kThreads == (kEpiWarps + 1 + kProdWarps) * 32, "warp roles");
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kProdTid0 = (kEpiWarps + 1) * 32;
constexpr int kMaxSlots = 32;
constexpr int kKc = 64;          // columns of the rank per job (128 bytes of a 16-bit row)
constexpr int kTileWords = 4;    // 128 rows per tile
constexpr int kTmemCols = 256;   // two accumulators of up to 96 columns, at 0 and 128

enum : uint32_t { kDetFull = 0x6100, kDetEmpty = 0x6200, kDetAccFull = 0x6300, kDetAccEmpty = 0x6400,
                  kDetDone = 0x6500, kDetAlign = 0x6600 };

}  // namespace sc

// BT: token columns per part (8, 16 or 32); B <= BT tokens are live.
template <typename T, int BT>
__global__ void __launch_bounds__(sc::kThreads, 1) k_score_mma(ScoreMmaArgs a) {
  using namespace sc;
  constexpr int N3 = (3 * BT + 15) / 16 * 16;  // MMA N: hi, mid, lo parts (rows p*BT + b), padded
  constexpr uint32_t kSlotA = 128 * 128;       // U tile (128 rows x 128 bytes)
  constexpr uint32_t kSlot = kSlotA + N3 * 128;
  extern __shared__ __align__(1024) unsigned char ring[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxSlots + 2 * 2 + 1];
  __shared__ uint32_t s_tmem;
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxSlots;
  uint64_t* accf = bars + 2 * kMaxSlots;
  uint64_t* acce = accf + 2;
  uint64_t* done = acce + 2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int f = a.f, r = a.r, W = a.W, B = a.B;
  if (smem_addr(ring) & 1023u) {  // swizzled tiles need 1024-byte alignment
    if (tid == 0) set_status(a.hdr, kStCapacity, kDetAlign);
    return;
  }
  const int G = gridDim.x;
  const int w_lo = (int)(((long long)W * blockIdx.x) / G), w_hi = (int)(((long long)W * (blockIdx.x + 1)) / G);
  const int nw = w_hi - w_lo;
  if (nw <= 0) return;  // the same for every thread of the block
  const int ntile = (nw + kTileWords - 1) / kTileWords;
  const int nkc = r / kKc;
  const int S = min(kMaxSlots, (int)(a.ring_bytes / kSlot));

  if (tid == 0) {
    for (int s = 0; s < kMaxSlots; ++s) {
      mbar_init(&full[s], kProdThreads);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], kEpiWarps * 32);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp > kMmaWarp) {
    // ---- copies: the tile's U rows (rows past d_ff are left out) and the
    // three parts of the tokens' hidden vectors, 64 columns of the rank per job
    const int p = tid - kProdTid0;
    const char* U = static_cast<const char*>(a.U);
    const char* H = static_cast<const char*>(a.h3);
    const size_t rowb = (size_t)r * sizeof(T);
    int s = 0, job = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = 0; t < ntile && ok; ++t) {
      const int row0 = (w_lo + t * kTileWords) * 32;
      const int rows = min(min(w_hi - (w_lo + t * kTileWords), kTileWords) * 32, f - row0);
      for (int j = 0; j < nkc; ++j, ++job) {
        if (job >= S && !mbar_wait(&empty[s], ph ^ 1u, a.hdr, a.wait_ns, kDetEmpty)) {
          ok = false;
          break;
        }
        unsigned char* sl = ring + (size_t)s * kSlot;
        const size_t off = (size_t)j * (kKc * sizeof(T));
        for (int e = p; e < rows * 8; e += kProdThreads) {
          const int rr = e >> 3, c = e & 7;
          cp_async16(sl + sw128_k(rr, c), U + (size_t)(row0 + rr) * rowb + off + c * 16);
        }
        for (int e = p; e < 3 * BT * 8; e += kProdThreads) {
          const int n = e >> 3, c = e & 7;
          cp_async16(sl + kSlotA + sw128_k(n, c), H + (size_t)n * rowb + off + c * 16);
        }
        cp_async_arrive_noinc(&full[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---- one thread issues the MMAs: tile t accumulates in buffer t % 2
    if (lane == 0) {
      const uint32_t id = idesc(IsBf16<T>::v, 0, N3);
      const uint32_t ring_a = smem_addr(ring);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const int buf = t & 1;
        if (t >= 2 && !mbar_wait(&acce[buf], (uint32_t)((t >> 1) - 1) & 1u, a.hdr, a.wait_ns, kDetAccEmpty)) break;
        tc_fence_after();
        const uint32_t dt = tmem + buf * 128;
        for (int j = 0; j < nkc; ++j) {
          if (!mbar_wait(&full[s], ph, a.hdr, a.wait_ns, kDetFull)) {
            ok = false;
            break;
          }
          proxy_fence();
          tc_fence_after();
          const uint32_t sl = ring_a + (uint32_t)s * kSlot;
#pragma unroll
          for (int kk = 0; kk < kKc / 16; ++kk)
            mma(dt, sdesc_sw128(sl + kk * 32, 16, 1024), sdesc_sw128(sl + kSlotA + kk * 32, 16, 1024), id,
                (j | kk) != 0);
          mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) mma_commit(&accf[buf]);
      }
      mma_commit(done);
      mbar_wait(done, 0u, a.hdr, a.wait_ns, kDetDone);
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread m holds row m of the tile (tensor-memory lane m)
    const int m = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int t = 0; t < ntile; ++t) {
      const int buf = t & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&accf[buf], (uint32_t)(t >> 1) & 1u, a.hdr, a.wait_ns, kDetAccFull)))
        break;
      tc_fence_after();
      const int wt = w_lo + t * kTileWords;               // first word of the tile
      const int nwt = min(w_hi - wt, kTileWords);         // words of the tile
      const int row = wt * 32 + m;
      const bool valid = warp < nwt && row < f;
      const float bias = valid ? __ldg(a.pb + row) : 0.f;
      const uint32_t acc_t = tmem + lane_base + buf * 128;
      uint32_t words = 0;  // lane b ends up holding token b's word
#pragma unroll
      for (int c = 0; c < BT; c += 16) {
        float hi[16], mid[16], lo[16];
        tmem_ld16(acc_t + c, hi);
        tmem_ld16(acc_t + BT + c, mid);
        tmem_ld16(acc_t + 2 * BT + c, lo);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16 && c + q < BT; ++q) {
          const float sv = hi[q] + (mid[q] + lo[q]) + bias;
          const uint32_t wv = __ballot_sync(0xffffffffu, valid && c + q < B && sv > a.tau);
          if (lane == c + q) words = wv;
        }
      }
      tc_fence_before();
      mbar_arrive(&acce[buf]);
      if (warp < nwt && lane < B) a.mask[(size_t)lane * W + wt + warp] = words;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <typename T, int BT>
cudaError_t score_mma_launch(const ScoreMmaArgs& a, int grid, size_t smem, cudaStream_t s) {
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_score_mma<T, BT>, smem, &cur);
  if (e != cudaSuccess) return e;
  k_score_mma<T, BT><<<grid, sc::kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t score_mma_dispatch(const ScoreMmaArgs& a, int bt, int grid, size_t smem, cudaStream_t s) {
  switch (bt) {
    case 8: return score_mma_launch<T, 8>(a, grid, smem, s);
    case 16: return score_mma_launch<T, 16>(a, grid, smem, s);
    case 32: return score_mma_launch<T, 32>(a, grid, smem, s);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace sffn
