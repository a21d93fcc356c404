// Batched decode (up to 32 tokens) over the union of the tokens' predicted-
// active neurons, on the fifth-generation tensor cores (tcgen05, accumulators
// in tensor memory).
//
// Activation sparsity is per token, so a batch must read every row that any of
// its tokens needs, and the saving shrinks as the batch grows (sparsity page,
// "工程影響" / engineering impact, throughput paragraph; PowerInfer's own batch
// results under "批次大小影響" / batch-size impact).  Each token still keeps
// only its own neurons: a_{b,i} is zero unless neuron i is in token b's mask.
// Over the union the gathered rows form dense blocks, so the two products are
// tensor-core contractions:
//   GEMM1  D1[i][b]  = W_up[i] . x_b   (and W_gate[i] . x_b for ReGLU)
//   a[i][b]          = ReLU(D1 + b_i) or ReLU(Dg + b_i) * Du, masked by token
//   GEMM2  Y^T[j][b] = sum_i W_downT[i][j] a[i][b]
//
// Layout of the work.  The union's members, in ascending order, are dealt to
// the blocks in equal contiguous rank ranges (every block computes the union
// itself from the mask words, so no extra pass is needed).  A block's members
// form tiles of at most 128 neurons; per tile:
//   * GEMM1 jobs: 64 columns of d each, the gathered rows of W_up (W_gate) and
//     the tokens copied into a shared-memory slot, M = 128 neurons, N = token
//     columns, K = 64;
//   * epilogue: D1 read from tensor memory, activation and token mask applied,
//     a split into a 16-bit high part and a 16-bit remainder (so that the
//     second product keeps fp32-level accuracy) and stored as GEMM2's B operand;
//   * GEMM2 jobs: 128 rows of d each, the tile's W_downT rows (M = 128 output
//     rows, K = the tile's neurons, N = 2 x token columns); the result is read
//     from tensor memory and added into y with float atomics.
// Warp roles: warps 0-3 epilogue (tensor-memory lanes 0-127), warp 4 issues the
// MMAs (one thread) and owns the tensor-memory allocation, warps 5-12 copy rows
// with per-thread 16-byte cp.async into a ring of slots whose mbarriers count
// one arrival per copying thread.
//
// Shared-memory operand layouts.  Copied operands use the tensor cores'
// 128-byte swizzled layouts, so that every 128-byte line a copy brings in
// lands in 128 contiguous bytes of shared memory (the 16-byte pieces permuted
// by the row index):
//   GEMM1 A (gathered W_up / W_gate rows) and B (tokens): K-major, one 128-byte
//     row per neuron / token (64 elements of d), 8-row groups 1024 bytes apart;
//   GEMM2 A (gathered W_downT rows, 128 elements of d): MN-major, the two
//     64-element halves of d K2*128 bytes apart, rows in 1024-byte groups of 8.
// GEMM2 B (the activations, written by the epilogue) is not swizzled: K-major
// 8x16-byte core matrices, element (n, k) at (k/8)*LBO + n*16 + (k%8)*2, with
// LBO = N*16 + 16 so that the 2-byte stores of neighbouring lanes spread over
// the banks.

#pragma once

#include "kernels.cuh"
#include "tcgen05.cuh"

namespace sffn {
namespace un {

using namespace tc;

constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarps = 8;
constexpr int kThreads = kUnionThreads;
static_assert(kThreads == (kEpiWarps + 1 + kProdWarps) * 32, "warp roles");
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kProdTid0 = (kEpiWarps + 1) * 32;
constexpr int kMaxSlots = kUnionMaxSlots;
constexpr int kMaxAcc = 8;        // GEMM2 accumulators in flight, at most
constexpr int kKc = 64;           // columns of d per GEMM1 job (one 128-byte line per 16-bit row)
constexpr int kDTile = 128;       // rows of d per GEMM2 job
constexpr int kMaxTile = 128;     // neurons per tile (the MMA's M)
constexpr int kPieces = 8;        // 16-byte pieces a copying thread owns per job (2 x 128 rows x 8 / 256)
constexpr int kMaxWpt = kUnionMaxWpt;  // mask words per thread in the union scan
constexpr int kTmemCols = 512;
constexpr int kColUp = 0, kColGate = 32, kColAcc = 64;  // GEMM2 accumulators from column 64 on
constexpr int kXPieces = 4;       // token pieces a copying thread owns per job (up to 4 x 32 x 8 / 256)
constexpr size_t kAtBytes = kUnionAtBytes;

// Detail codes of the device status word (which wait gave up).
enum : uint32_t { kDetFull = 0x5100, kDetEmpty = 0x5200, kDetD1 = 0x5300, kDetAt = 0x5400,
                  kDetAccFull = 0x5500, kDetAccEmpty = 0x5600, kDetDone = 0x5700,
                  kDetAlign = 0x5800 };

// Job order of block-dependent rotation: block b starts its walk over the
// n column chunks at chunk `o`, so that the blocks do not all read the same
// token columns or add into the same output rows at the same moment.
__device__ __forceinline__ int rot(int j, int o, int n) {
  const int v = j + o;
  return v >= n ? v - n : v;
}

// Rows of tile t when n members are split into nt near-equal tiles.
__device__ __forceinline__ int tile_begin(int t, int n, int nt) { return (int)(((long long)t * n) / nt); }

}  // namespace un

// BT: token columns of the tiles (8, 16 or 32); B <= BT tokens are live.
template <typename T, int BT>
__global__ void __launch_bounds__(un::kThreads, 1) k_union(UnionArgs a) {
  using namespace un;
  constexpr int N1 = BT < 16 ? 16 : BT;  // GEMM1 token columns (M = 128 needs N % 16 == 0)
  constexpr int N2 = 2 * BT;             // GEMM2 columns: high parts, then remainders
  constexpr int kLa = N2 * 16 + 16;      // activation operand: stride of its 8-neuron core-matrix blocks
  constexpr int kNAcc = (kTmemCols - kColAcc) / N2 < kMaxAcc ? (kTmemCols - kColAcc) / N2 : kMaxAcc;
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(1024) unsigned char dsm[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxSlots + 2 * kMaxAcc + 3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_scan[kWarps];
  __shared__ int s_nwords;
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxSlots;
  uint64_t* accf = bars + 2 * kMaxSlots;
  uint64_t* acce = accf + kMaxAcc;
  uint64_t* d1f = acce + kMaxAcc;
  uint64_t* atr = d1f + 1;
  uint64_t* done = atr + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, d = a.d, W = a.W;
  if (smem_addr(dsm) & 1023u) {  // swizzled tiles need 1024-byte alignment
    if (tid == 0) set_status(a.hdr, kStCapacity, kDetAlign);
    return;
  }
  const int nm = a.act == kReglu ? 2 : 1;
  unsigned char* ring = dsm;
  unsigned char* at = dsm + a.ring_bytes;
  int32_t* nidx = reinterpret_cast<int32_t*>(at + kAtBytes);
  uint32_t* tbits = reinterpret_cast<uint32_t*>(nidx + a.list_cap);
  float* nbias = reinterpret_cast<float*>(tbits + a.list_cap);
  int2* wlist = reinterpret_cast<int2*>(at);  // scratch until the first epilogue

  // ---- 1. union of the token masks, its size, and this block's rank range
  const int wpt = (W + kThreads - 1) / kThreads;
  const int w0 = tid * wpt;
  uint32_t uw[kMaxWpt];
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < kMaxWpt; ++q) {
    uint32_t u = 0;
    const int w = w0 + q;
    if (q < wpt && w < W) {
#pragma unroll
      for (int bb = 0; bb < BT; ++bb)
        if (bb < B) u |= __ldcg(a.mask + (size_t)bb * W + w);
    }
    uw[q] = u;
    cnt += __popc(u);
  }
  if (tid == 0) s_nwords = 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int excl = incl - cnt, total = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    const int v = s_scan[i];
    if (i < warp) excl += v;
    total += v;
  }
  const int G = gridDim.x;
  const int lo = (int)(((long long)total * blockIdx.x) / G);
  const int hi = (int)(((long long)total * (blockIdx.x + 1)) / G);
  const int nc = hi - lo;
  if (nc == 0) return;  // the same for every thread of the block

  // words holding this block's members, then one warp per word: lane b holds
  // token b's word, and a ballot per bit turns it into that neuron's token bits
  {
    int rank = excl;
#pragma unroll
    for (int q = 0; q < kMaxWpt; ++q) {
      const int pc = __popc(uw[q]);
      if (pc > 0 && rank < hi && rank + pc > lo) wlist[atomicAdd(&s_nwords, 1)] = make_int2(w0 + q, rank);
      rank += pc;
    }
  }
  __syncthreads();
  const int nwords = s_nwords;
  for (int i = warp; i < nwords; i += kWarps) {
    const int2 wr = wlist[i];
    const uint32_t tw = lane < B ? __ldcg(a.mask + (size_t)lane * W + wr.x) : 0u;
    const uint32_t u = __reduce_or_sync(0xffffffffu, tw);
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t bj = __ballot_sync(0xffffffffu, (tw >> j) & 1u);
      if (lane == j) mine = bj;
    }
    if ((u >> lane) & 1u) {
      const int rank = wr.y + __popc(u & ((1u << lane) - 1u));
      if (rank >= lo && rank < hi) {
        const int neuron = wr.x * 32 + lane;
        nidx[rank - lo] = neuron;
        tbits[rank - lo] = mine;
        nbias[rank - lo] = a.b != nullptr ? __ldg(a.b + neuron) : 0.f;
      }
    }
  }

  // ---- 2. tiles and jobs.  A block's members form nt near-equal tiles of at
  // most 128 neurons.  A GEMM1 job covers KA column chunks of 64 (KA x 128
  // bytes of every gathered row), a GEMM2 job DA output tiles of 128 rows of d;
  // both widen when the tiles are short, so that every job moves enough bytes
  // to amortise its hand-offs.  A thread owns at most kPieces pieces per job.
  const int nk = d / kKc, nd = d / kDTile;
  const int nt = (nc + kMaxTile - 1) / kMaxTile;
  const int rmax = (nc + nt - 1) / nt;
  const int r8max = (rmax + 7) & ~7, k2max = (rmax + 15) & ~15;
  int KA = 1, DA = 1;
  while (KA < 4 && 2 * KA * nm * r8max <= kPieces * kProdThreads / 8 && nk % (2 * KA) == 0) KA *= 2;
  while (DA < 4 && 2 * DA * k2max <= kPieces * kProdThreads / 16 && nd % (2 * DA) == 0 && 2 * DA <= kNAcc / 2) DA *= 2;
  const uint32_t slot_bytes =
      ((uint32_t)max(KA * (nm * r8max + N1) * 128, DA * k2max * 256) + 1023u) & ~1023u;
  // Tiles of at most 64 neurons use M = 64 MMAs for GEMM1: half the operand
  // bytes per MMA (the tensor core reads every one of the M rows).
  const bool m64 = r8max <= 64;
  const int S = min(kMaxSlots, (int)(a.ring_bytes / slot_bytes));
  // W_downT rows past a tile's end (up to the next 16) are read by GEMM2
  // against zero activations, so they must hold finite values: zero them once
  // in every slot (copies only ever write weights and tokens there).
  for (int t = 0; t < nt; ++t) {
    const int R = tile_begin(t + 1, nc, nt) - tile_begin(t, nc, nt);
    const int K2 = (R + 15) & ~15, pad = K2 - R;
    for (int e = tid; e < S * DA * 16 * pad; e += kThreads) {  // 16 pieces of 16 bytes per padded row
      const int s = e / (DA * 16 * pad), rem = e - s * DA * 16 * pad, q = rem / (16 * pad),
                rem2 = rem - q * 16 * pad, k = R + rem2 / 16, c16 = rem2 & 15;
      *reinterpret_cast<uint4*>(ring + (size_t)s * slot_bytes + q * K2 * 256 + sw128_mn(k, c16, K2)) =
          make_uint4(0, 0, 0, 0);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kMaxSlots; ++s) {
      mbar_init(&full[s], kProdThreads);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kNAcc; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], kEpiWarps * 32);
    }
    mbar_init(d1f, 1);
    mbar_init(atr, kEpiWarps * 32);
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
  const int off1 = (int)((blockIdx.x * 7u) % (unsigned)nk), off2 = (int)((blockIdx.x * 5u) % (unsigned)nd);

  if (warp > kMmaWarp) {
    // ---- 3a. copies: GEMM1 jobs (columns of the tile's W_up/W_gate rows and
    // of the tokens), then GEMM2 jobs (columns of its W_downT rows).  A thread
    // copies the same pieces of the same rows in every job of a phase, so their
    // addresses are formed once per tile; only the column offset moves.
    const int p = tid - kProdTid0;
    const char* xg = static_cast<const char*>(a.x);
    const char* wu = static_cast<const char*>(a.w_up);
    const char* wg = static_cast<const char*>(a.w_gate);
    const char* wd = static_cast<const char*>(a.w_downT);
    const size_t rowb = (size_t)d * sizeof(T);
    int s = 0, job = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = 0; t < nt && ok; ++t) {
      const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
      const int R8 = (R + 7) & ~7, K2 = (R + 15) & ~15;
      const uint32_t blk = (uint32_t)(nm * R8 + N1) * 128;  // one column chunk of the tile's rows and tokens
      const int32_t* ti = nidx + r0;
      const char* src[kPieces];
      uint32_t dst[kPieces];
      int sub[kPieces];
      int np = 0;
      const int per_atom = nm * R * 8;
#pragma unroll
      for (int q = 0; q < kPieces; ++q) {  // 8 pieces of 16 bytes per row, matrix and column chunk
        const int e = p + q * kProdThreads;
        src[q] = nullptr;
        dst[q] = 0;
        sub[q] = 0;
        if (e < KA * per_atom) {
          const int at_i = e / per_atom, rem = e - at_i * per_atom;
          const int m = rem >= R * 8 ? 1 : 0, rem2 = rem - m * R * 8, r = rem2 >> 3, c = rem2 & 7;
          src[q] = (m ? wg : wu) + (size_t)ti[r] * a.wstride + c * 16;
          dst[q] = at_i * blk + sw128_k(m * R8 + r, c);
          sub[q] = at_i;
          np = q + 1;
        }
      }
      const char* srcx[kXPieces];
      uint32_t dstx[kXPieces];
      int subx[kXPieces];
      int nx = 0;
#pragma unroll
      for (int q = 0; q < kXPieces; ++q) {
        const int e = p + q * kProdThreads;
        srcx[q] = nullptr;
        dstx[q] = 0;
        subx[q] = 0;
        if (e < KA * B * 8) {
          const int at_i = e / (B * 8), rem = e - at_i * B * 8, n = rem >> 3, c = rem & 7;
          srcx[q] = xg + (size_t)n * rowb + c * 16;
          dstx[q] = at_i * blk + sw128_k(nm * R8 + n, c);
          subx[q] = at_i;
          nx = q + 1;
        }
      }
      for (int j = 0; j < nk / KA; ++j, ++job) {
        if (job >= S && !mbar_wait(&empty[s], ph ^ 1u, a.hdr, a.wait_ns, kDetEmpty)) {
          ok = false;
          break;
        }
        unsigned char* sl = ring + (size_t)s * slot_bytes;
#pragma unroll
        for (int q = 0; q < kPieces; ++q)
          if (q < np) cp_async16(sl + dst[q], src[q] + (size_t)rot(j * KA + sub[q], off1, nk) * (kKc * sizeof(T)));
#pragma unroll
        for (int q = 0; q < kXPieces; ++q)
          if (q < nx) cp_async16(sl + dstx[q], srcx[q] + (size_t)rot(j * KA + subx[q], off1, nk) * (kKc * sizeof(T)));
        cp_async_arrive_noinc(&full[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      np = 0;
#pragma unroll
      for (int q = 0; q < kPieces; ++q) {  // 16 pieces of 16 bytes per row and output tile
        const int e = p + q * kProdThreads;
        src[q] = nullptr;
        dst[q] = 0;
        sub[q] = 0;
        if (e < DA * R * 16) {
          const int ot = e / (R * 16), rem = e - ot * R * 16, r = rem >> 4, c16 = rem & 15;
          src[q] = wd + (size_t)ti[r] * a.wstride + c16 * 16;
          dst[q] = ot * K2 * 256 + sw128_mn(r, c16, K2);
          sub[q] = ot;
          np = q + 1;
        }
      }
      for (int j = 0; j < nd / DA; ++j, ++job) {
        if (job >= S && !mbar_wait(&empty[s], ph ^ 1u, a.hdr, a.wait_ns, kDetEmpty)) {
          ok = false;
          break;
        }
        unsigned char* sl = ring + (size_t)s * slot_bytes;
#pragma unroll
        for (int q = 0; q < kPieces; ++q)
          if (q < np) cp_async16(sl + dst[q], src[q] + (size_t)rot(j * DA + sub[q], off2, nd) * (kDTile * sizeof(T)));
        cp_async_arrive_noinc(&full[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---- 3b. one thread issues every MMA
    if (lane == 0) {
      const uint32_t id1 = idesc(IsBf16<T>::v, 0, N1, m64 ? 64 : 128), id2 = idesc(IsBf16<T>::v, 1, N2);
      const uint32_t ring_a = smem_addr(ring), at_a = smem_addr(at);
      int s = 0, ac = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
        const int R8 = (R + 7) & ~7, K2 = (R + 15) & ~15;
        const uint32_t blk = (uint32_t)(nm * R8 + N1) * 128;
        for (int j = 0; j < nk / KA; ++j) {
          if (!mbar_wait(&full[s], ph, a.hdr, a.wait_ns, kDetFull)) {
            ok = false;
            break;
          }
          proxy_fence();
          tc_fence_after();
          const uint32_t sl = ring_a + (uint32_t)s * slot_bytes;
          for (int at_i = 0; at_i < KA; ++at_i) {
            const uint32_t wa = sl + at_i * blk, xa = wa + (uint32_t)(nm * R8) * 128;
#pragma unroll
            for (int kk = 0; kk < kKc / 16; ++kk) {  // a K step of 16 is 32 bytes inside the 128-byte rows
              const uint64_t bd = sdesc_sw128(xa + kk * 32, 16, 1024);
              const uint32_t acc = (j | at_i | kk) != 0;
              mma(tmem + kColUp, sdesc_sw128(wa + kk * 32, 16, 1024), bd, id1, acc);
              if (nm == 2) mma(tmem + kColGate, sdesc_sw128(wa + R8 * 128 + kk * 32, 16, 1024), bd, id1, acc);
            }
          }
          mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(d1f);
        if (!mbar_wait(atr, (uint32_t)t & 1u, a.hdr, a.wait_ns, kDetAt)) break;
        proxy_fence();
        tc_fence_after();
        for (int j = 0; j < nd / DA && ok; ++j) {
          if (!mbar_wait(&full[s], ph, a.hdr, a.wait_ns, kDetFull)) {
            ok = false;
            break;
          }
          proxy_fence();
          const uint32_t sl = ring_a + (uint32_t)s * slot_bytes;
          for (int ot = 0; ot < DA; ++ot, ++ac) {
            const int buf = ac % kNAcc;
            if (ac >= kNAcc &&
                !mbar_wait(&acce[buf], (uint32_t)((ac / kNAcc) - 1) & 1u, a.hdr, a.wait_ns, kDetAccEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dt = tmem + kColAcc + buf * N2, wa = sl + ot * K2 * 256;
            for (int kk = 0; kk < K2 / 16; ++kk)  // a K step of 16 rows is two 1024-byte row groups
              mma(dt, sdesc_sw128(wa + kk * 2048, K2 * 128, 1024), sdesc(at_a + kk * 2 * kLa, kLa, 128), id2, kk != 0);
            mma_commit(&accf[buf]);
          }
          mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      mma_commit(done);
      mbar_wait(done, 0u, a.hdr, a.wait_ns, kDetDone);
    }
    __syncwarp();
  } else {
    // ---- 3c. epilogue: warp w reads tensor-memory lanes [32w, 32w + 32).
    // GEMM1 row of this thread: its lane (M = 128), or with M = 64 lanes 0-15
    // of each warp hold rows 16w .. 16w + 15; GEMM2 row: its lane.
    const int m = tid;
    const int m1 = m64 ? (lane < 16 ? warp * 16 + lane : -1) : tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int ac = 0;
    for (int t = 0; t < nt; ++t) {
      const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
      const int K2 = (R + 15) & ~15;
      if (!__all_sync(0xffffffffu, mbar_wait(d1f, (uint32_t)t & 1u, a.hdr, a.wait_ns, kDetD1))) break;
      tc_fence_after();
      uint32_t tb = 0;
      float bias = 0.f;
      if (m1 >= 0 && m1 < R) {
        tb = tbits[r0 + m1];
        bias = nbias[r0 + m1];
      }
      unsigned char* col = at + (m1 >> 3) * kLa + (m1 & 7) * 2;
#pragma unroll
      for (int c = 0; c < N1; c += 16) {
        float u[16], g[16];
        tmem_ld16(tmem + lane_base + kColUp + c, u);
        if (nm == 2) tmem_ld16(tmem + lane_base + kColGate + c, g);
        tmem_wait_ld();
        if (m1 >= 0 && m1 < K2) {
#pragma unroll
          for (int q = 0; q < 16 && c + q < BT; ++q) {
            float av = 0.f;
            if ((tb >> (c + q)) & 1u) av = nm == 2 ? fmaxf(g[q] + bias, 0.f) * u[q] : fmaxf(u[q] + bias, 0.f);
            const T hi = from_float<T>(av);
            const T rem = from_float<T>(av - to_float<T>(hi));
            *reinterpret_cast<T*>(col + (c + q) * 16) = hi;
            *reinterpret_cast<T*>(col + (BT + c + q) * 16) = rem;
          }
        }
      }
      proxy_fence();
      tc_fence_before();
      mbar_arrive(atr);
      bool ok = true;
      for (int j = 0; j < nd; ++j, ++ac) {
        const int buf = ac % kNAcc;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&accf[buf], (uint32_t)(ac / kNAcc) & 1u, a.hdr, a.wait_ns, kDetAccFull))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc_t = tmem + lane_base + kColAcc + buf * N2;
        float* yr = a.y + (size_t)rot(j, off2, nd) * kDTile + m;
#pragma unroll
        for (int c = 0; c < BT; c += 16) {
          float vh[16], vl[16];
          tmem_ld16(acc_t + c, vh);
          tmem_ld16(acc_t + BT + c, vl);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 16 && c + q < BT; ++q)
            if (c + q < B) atomicAdd(yr + (size_t)(c + q) * d, vh[q] + vl[q]);
        }
        tc_fence_before();
        mbar_arrive(&acce[buf]);
      }
      if (!ok) break;
    }
  }

  // ---- 4. every MMA has completed (the issuing thread waited for it) and
  // every tensor-memory read is done: release the columns
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <typename T, int BT>
cudaError_t union_launch(const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  static int cur = 48 * 1024;
  const cudaError_t e = ensure_dyn_smem(k_union<T, BT>, cfg.smem, &cur);
  if (e != cudaSuccess) return e;
  k_union<T, BT><<<grid, un::kThreads, cfg.smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t union_dispatch(const UnionConfig& cfg, const UnionArgs& a, int grid, cudaStream_t s) {
  switch (cfg.bt) {
    case 8: return union_launch<T, 8>(cfg, a, grid, s);
    case 16: return union_launch<T, 16>(cfg, a, grid, s);
    case 32: return union_launch<T, 32>(cfg, a, grid, s);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace sffn
