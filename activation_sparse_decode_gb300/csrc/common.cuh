// Device helpers shared by the sparse-FFN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sffn {

// Device status codes (values of sffn_status).
enum : uint32_t { kStOk = 0, kStCapacity = 4, kStTimeout = 5 };

// Header at offset 0 of every workspace (256 bytes).
struct WsHeader {
  uint32_t status;     // first device-side error (sticky until read)
  uint32_t detail;     // where it happened (kernel-specific code)
  uint32_t bar_count;  // grid barrier: arrivals in the current generation
  uint32_t reserved;
  unsigned long long arrivals;  // layer kernel: launch counter (one per block, rounded up to 2^20 per launch)
  uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum Act : int { kRelu = 0, kReglu = 1 };

// ---------------------------------------------------------------- dtype chunks
// Every row is processed in 16-byte chunks: 4 fp32 or 8 fp16/bf16 values.
template <typename T> struct Chunk;
template <> struct Chunk<float> { static constexpr int N = 4; };
template <> struct Chunk<__half> { static constexpr int N = 8; };
template <> struct Chunk<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ void unpack(const uint4& u, float* o);

template <>
__device__ __forceinline__ void unpack<float>(const uint4& u, float* o) {
  o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
  o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack<__half>(const uint4& u, float* o) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 f = __half22float2(h);
    o[2 * i] = f.x; o[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4& u, float* o) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { o[2 * i] = bf16lo(w[i]); o[2 * i + 1] = bf16hi(w[i]); }
}

template <typename T> __device__ __forceinline__ T from_float(float v);
template <> __device__ __forceinline__ float from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_float<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 16-byte global load through the read-only path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- timing / status
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first device-side error; later ones are dropped.
__device__ __forceinline__ void set_status(WsHeader* h, uint32_t code, uint32_t detail) {
  if (atomicCAS(&h->status, 0u, code) == 0u) atomicExch(&h->detail, detail);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier over `expected` resident blocks.
//
// Every block has its own release flag, flags[b * 32] (one 128-byte line
// each); all flags hold the same generation.  A block learns that generation
// before it can change -- at kernel start, barrier_generation() -- so arriving
// costs one round trip: an acq_rel atomic add on the shared counter.  The last
// block to arrive resets the counter, fences once, and stores generation + 1
// into every flag; the others poll only their own line, so no two blocks poll
// the same line and the release stores do not queue behind pollers.  `gen` is
// the generation this barrier waits to leave (the next barrier of the same
// launch waits on gen + 1).
//
// One thread of the block (`bthread`) does the arrival, the release and the
// wait.  Every wait is bounded: after limit_ns the block records kStTimeout
// and returns false (the counter is then left mid-count; zero the workspace
// before reusing it).  All threads of the block must call it.
__host__ __device__ constexpr size_t barrier_flag_bytes(uint32_t blocks) { return (size_t)blocks * 128; }

__device__ __forceinline__ uint32_t barrier_generation(const uint32_t* flags) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flags + (size_t)blockIdx.x * 32) : "memory");
  return v;
}

// The warp-level part, called by all 32 lanes of one warp: lane 0 arrives;
// if it was the last block, the counter is reset and the 32 lanes store the
// next generation into the flags (a few stores each, each lane fencing first);
// otherwise lane 0 waits on its own flag.  Returns the same value on all lanes.
__device__ __forceinline__ bool barrier_arrive_wait_warp(WsHeader* h, uint32_t* flags, uint32_t expected,
                                                         uint32_t gen, uint64_t limit_ns, uint32_t detail) {
  const uint32_t lane = threadIdx.x & 31u;
  uint32_t old = 0;
  if (lane == 0)
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(&h->bar_count) : "memory");
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == expected - 1) {
    if (lane == 0)  // nobody touches the counter again before the release below
      asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(&h->bar_count) : "memory");
    __syncwarp();
    __threadfence();  // the reset and everything this block saw precede the release
    for (uint32_t b = lane; b < expected; b += 32)
      asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flags + (size_t)b * 32), "r"(gen + 1u) : "memory");
    return true;
  }
  int ok = 1;
  if (lane == 0) {
    const uint32_t* mine = flags + (size_t)blockIdx.x * 32;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(mine) == gen) {
      if (globaltimer_ns() - t0 > limit_ns) {
        set_status(h, kStTimeout, detail);
        ok = 0;
        break;
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}


// Whole-block form; warp `bwarp` does the barrier work.
__device__ __forceinline__ bool grid_barrier(WsHeader* h, uint32_t* flags, uint32_t expected, uint32_t gen,
                                             uint64_t limit_ns, uint32_t detail, uint32_t bwarp = 0) {
  __shared__ int s_ok;
  __syncthreads();
  if ((threadIdx.x >> 5) == bwarp) {
    const bool ok = barrier_arrive_wait_warp(h, flags, expected, gen, limit_ns, detail);
    if ((threadIdx.x & 31) == 0) s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase; false (and kStTimeout) if it never completes.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, WsHeader* h,
                                          uint64_t limit_ns, uint32_t detail) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      set_status(h, kStTimeout, detail);
      return false;
    }
  }
  return true;
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory, completing
// on `bar` with a byte count.  dst, src and bytes must be 16-byte aligned.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Per-thread 16-byte asynchronous copy global -> shared (L1 bypassed), many in
// flight per thread without registers; completion per thread via wait_all.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The mbarrier receives one arrival once every cp.async this thread issued
// before it has landed (the barrier's expected count includes the arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch: wait until the preceding kernel on the stream
// has completed and its memory is visible (a no-op when the launch was not
// programmatic), and allow the next kernel to begin launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Thread-block clusters: this block's rank, a full cluster barrier (every
// thread of every block of the cluster; release/acquire order shared memory
// across the cluster), and loads from a peer block's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Split form of the cluster barrier: an arrival that orders nothing (the
// caller has consumed every value it read from other members), and the wait.
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_peer_v2(uint32_t addr, int x, int y) {
  asm volatile("st.shared::cluster.v2.s32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}
// Arrive (release, cluster scope) on an mbarrier in another block of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Test (acquire, cluster scope) whether the phase with `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ void st_peer_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t peer_smem(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Raises a kernel's dynamic shared-memory limit when a launch needs more than
// any earlier launch of it did (`cur` is that kernel's high-water mark).
template <typename F>
inline cudaError_t ensure_dyn_smem(F* func, size_t bytes, int* cur) {
  if ((int)bytes <= *cur) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *cur = (int)bytes;
  return e;
}

}  // namespace sffn
