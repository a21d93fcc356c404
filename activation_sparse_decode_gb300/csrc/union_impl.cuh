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
// Shared-memory operand layouts (no swizzle; 8x16-byte core matrices):
//   K-major  (GEMM1 A and B, GEMM2 B): element (row, k) at
//            (k/8)*LBO + row*16 + (k%8)*2, LBO = rows*16, SBO = 128;
//   MN-major (GEMM2 A = W_downT rows): element (m, k) at
//            (m/8)*SBO + k*16 + (m%8)*2, LBO = 128 (next 8 k), SBO = K*16.

#pragma once

#include "kernels.cuh"

namespace sffn {
namespace un {

constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarps = 8;
constexpr int kThreads = kUnionThreads;
static_assert(kThreads == (kEpiWarps + 1 + kProdWarps) * 32, "warp roles");
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kProdTid0 = (kEpiWarps + 1) * 32;
constexpr int kMaxSlots = kUnionMaxSlots;
constexpr int kNAcc = 4;          // GEMM2 accumulators in flight
constexpr int kKc = 64;           // columns of d per GEMM1 job (one 128-byte line per 16-bit row)
constexpr int kDTile = 128;       // rows of d per GEMM2 job
constexpr int kMaxTile = 128;     // neurons per tile (the MMA's M)
constexpr int kMaxWpt = kUnionMaxWpt;  // mask words per thread in the union scan
constexpr int kTmemCols = 512;
constexpr int kColUp = 0, kColGate = 32, kColAcc = 64, kAccStride = 64;
constexpr size_t kAtBytes = kUnionAtBytes;

// Detail codes of the device status word (which wait gave up).
enum : uint32_t { kDetFull = 0x5100, kDetEmpty = 0x5200, kDetD1 = 0x5300, kDetAt = 0x5400,
                  kDetAccFull = 0x5500, kDetAccEmpty = 0x5600, kDetDone = 0x5700 };

// tcgen05 shared-memory matrix descriptor, no swizzle (version field = 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind::f16 with fp32 accumulation, M = 128.
__device__ __forceinline__ uint32_t idesc(int bf16, int a_mn_major, int n) {
  return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kMaxTile >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival once every MMA this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T> __device__ __forceinline__ float to_float(T v);
template <> __device__ __forceinline__ float to_float<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Rows of tile t when n members are split into nt near-equal tiles.
__device__ __forceinline__ int tile_begin(int t, int n, int nt) { return (int)(((long long)t * n) / nt); }

}  // namespace un

// BT: token columns of the tiles (8, 16 or 32); B <= BT tokens are live.
template <typename T, int BT>
__global__ void __launch_bounds__(un::kThreads, 1) k_union(UnionArgs a) {
  using namespace un;
  constexpr int N1 = BT < 16 ? 16 : BT;  // GEMM1 token columns (M = 128 needs N % 16 == 0)
  constexpr int N2 = 2 * BT;             // GEMM2 columns: high parts, then remainders
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(1024) unsigned char dsm[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxSlots + 2 * kNAcc + 3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_scan[kWarps];
  __shared__ int s_nwords;
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxSlots;
  uint64_t* accf = bars + 2 * kMaxSlots;
  uint64_t* acce = accf + kNAcc;
  uint64_t* d1f = acce + kNAcc;
  uint64_t* atr = d1f + 1;
  uint64_t* done = atr + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, d = a.d, W = a.W;
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

  // ---- 2. tiles, slots; W_downT rows past a tile's end (up to the next 16)
  // are read by GEMM2 against zero activations, so they must hold finite
  // values: zero them once in every slot (copies only ever write weights).
  const int nt = (nc + kMaxTile - 1) / kMaxTile;
  const int rmax = (nc + nt - 1) / nt;
  const int r8max = (rmax + 7) & ~7, k2max = (rmax + 15) & ~15;
  const uint32_t slot_bytes =
      ((uint32_t)max(nm * r8max * 128 + N1 * 128, k2max * 256) + 127u) & ~127u;
  const int S = min(kMaxSlots, (int)(a.ring_bytes / slot_bytes));
  for (int t = 0; t < nt; ++t) {
    const int R = tile_begin(t + 1, nc, nt) - tile_begin(t, nc, nt);
    const int K2 = (R + 15) & ~15, pad = K2 - R;
    for (int e = tid; e < S * 16 * pad; e += kThreads) {
      const int s = e / (16 * pad), rem = e - s * 16 * pad, g = rem / pad, k = R + (rem - g * pad);
      *reinterpret_cast<uint4*>(ring + (size_t)s * slot_bytes + g * (K2 * 16) + k * 16) = make_uint4(0, 0, 0, 0);
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
  const int nk = d / kKc, nd = d / kDTile;

  if (warp > kMmaWarp) {
    // ---- 3a. copies: GEMM1 jobs (W_up/W_gate columns [k0, k0+64) of the
    // tile's rows, and the tokens), then GEMM2 jobs (W_downT columns [d0, d0+128))
    const int p = tid - kProdTid0;
    const T* xg = static_cast<const T*>(a.x);
    const T* wu = static_cast<const T*>(a.w_up);
    const T* wg = static_cast<const T*>(a.w_gate);
    const T* wd = static_cast<const T*>(a.w_downT);
    int s = 0, job = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = 0; t < nt && ok; ++t) {
      const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
      const int R8 = (R + 7) & ~7, K2 = (R + 15) & ~15;
      const int32_t* ti = nidx + r0;
      for (int j = 0; j < nk + nd; ++j, ++job) {
        if (job >= S && !mbar_wait(&empty[s], ph ^ 1u, a.hdr, a.wait_ns, kDetEmpty)) {
          ok = false;
          break;
        }
        unsigned char* sl = ring + (size_t)s * slot_bytes;
        if (j < nk) {
          const int k0 = j * kKc;
          for (int m = 0; m < nm; ++m) {
            const T* wmat = m == 0 ? wu : wg;
            unsigned char* dst = sl + m * R8 * 128;
            for (int e = p; e < R * 8; e += kProdThreads) {
              const int r = e >> 3, c = e & 7;
              cp_async16(dst + c * (R8 * 16) + r * 16, wmat + (size_t)ti[r] * d + k0 + c * 8);
            }
          }
          if (p < B * 8) {
            const int n = p >> 3, c = p & 7;
            cp_async16(sl + nm * R8 * 128 + c * (N1 * 16) + n * 16, xg + (size_t)n * d + k0 + c * 8);
          }
        } else {
          const int d0 = (j - nk) * kDTile;
          for (int e = p; e < R * 16; e += kProdThreads) {
            const int r = e >> 4, g = e & 15;
            cp_async16(sl + g * (K2 * 16) + r * 16, wd + (size_t)ti[r] * d + d0 + g * 8);
          }
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
    // ---- 3b. one thread issues every MMA
    if (lane == 0) {
      const uint32_t id1 = idesc(IsBf16<T>::v, 0, N1), id2 = idesc(IsBf16<T>::v, 1, N2);
      const uint32_t ring_a = smem_addr(ring), at_a = smem_addr(at);
      int s = 0, ac = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
        const int R8 = (R + 7) & ~7, K2 = (R + 15) & ~15;
        for (int j = 0; j < nk; ++j) {
          if (!mbar_wait(&full[s], ph, a.hdr, a.wait_ns, kDetFull)) {
            ok = false;
            break;
          }
          proxy_fence();
          tc_fence_after();
          const uint32_t sl = ring_a + (uint32_t)s * slot_bytes;
          const uint32_t xa = sl + nm * R8 * 128;
#pragma unroll
          for (int kk = 0; kk < kKc / 16; ++kk) {
            const uint64_t bd = sdesc(xa + kk * 2 * N1 * 16, N1 * 16, 128);
            const uint32_t acc = (j | kk) != 0;
            mma(tmem + kColUp, sdesc(sl + kk * 2 * R8 * 16, R8 * 16, 128), bd, id1, acc);
            if (nm == 2) mma(tmem + kColGate, sdesc(sl + R8 * 128 + kk * 2 * R8 * 16, R8 * 16, 128), bd, id1, acc);
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
        for (int j = 0; j < nd; ++j, ++ac) {
          const int buf = ac % kNAcc;
          if (!mbar_wait(&full[s], ph, a.hdr, a.wait_ns, kDetFull) ||
              (ac >= kNAcc && !mbar_wait(&acce[buf], (uint32_t)((ac / kNAcc) - 1) & 1u, a.hdr, a.wait_ns,
                                         kDetAccEmpty))) {
            ok = false;
            break;
          }
          proxy_fence();
          tc_fence_after();
          const uint32_t sl = ring_a + (uint32_t)s * slot_bytes;
          const uint32_t dt = tmem + kColAcc + buf * kAccStride;
          for (int kk = 0; kk < K2 / 16; ++kk)
            mma(dt, sdesc(sl + kk * 256, 128, K2 * 16), sdesc(at_a + kk * 2 * N2 * 16, N2 * 16, 128), id2, kk != 0);
          mma_commit(&empty[s]);
          mma_commit(&accf[buf]);
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
    // ---- 3c. epilogue: warp w reads tensor-memory lanes [32w, 32w + 32)
    const int m = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int ac = 0;
    for (int t = 0; t < nt; ++t) {
      const int r0 = tile_begin(t, nc, nt), R = tile_begin(t + 1, nc, nt) - r0;
      const int K2 = (R + 15) & ~15;
      if (!__all_sync(0xffffffffu, mbar_wait(d1f, (uint32_t)t & 1u, a.hdr, a.wait_ns, kDetD1))) break;
      tc_fence_after();
      uint32_t tb = 0;
      float bias = 0.f;
      if (m < R) {
        tb = tbits[r0 + m];
        bias = nbias[r0 + m];
      }
      unsigned char* col = at + (m >> 3) * (N2 * 16) + (m & 7) * 2;
#pragma unroll
      for (int c = 0; c < N1; c += 16) {
        float u[16], g[16];
        tmem_ld16(tmem + lane_base + kColUp + c, u);
        if (nm == 2) tmem_ld16(tmem + lane_base + kColGate + c, g);
        tmem_wait_ld();
        if (m < K2) {
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
        const uint32_t acc_t = tmem + lane_base + kColAcc + buf * kAccStride;
        float* yr = a.y + (size_t)j * kDTile + m;
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
