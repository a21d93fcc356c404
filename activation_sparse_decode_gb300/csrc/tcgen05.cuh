// tcgen05 building blocks shared by the tensor-core kernels (sm_103a):
// shared-memory matrix descriptors, the kind::f16 instruction descriptor,
// MMA issue and commit, tensor-memory loads, fences, and the 128-byte swizzled
// operand layouts the copies write.
#pragma once

#include "common.cuh"

namespace sffn {
namespace tc {

// tcgen05 shared-memory matrix descriptor, no swizzle (version field = 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind::f16 with fp32 accumulation (M = 128 or 64).
// With M = 64 the accumulator's row m sits in tensor-memory lane
// (m / 16) * 32 + m % 16: 16 rows in each warp's quarter of the lanes.
__device__ __forceinline__ uint32_t idesc(int bf16, int a_mn_major, int n, int m = 128) {
  return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
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


// Shared-memory matrix descriptor with 128-byte swizzling (layout type 2).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return sdesc(addr, lbo, sbo) | (2ull << 61);
}

// 128-byte-swizzled K-major tile: row `row` is 128 contiguous bytes (64
//16-bit elements of K); its 16-byte piece c sits at position c ^ (row % 8).
// Tiles start on 1024-byte boundaries (8 rows).
__device__ __forceinline__ uint32_t sw128_k(int row, int c) {
  return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4));
}

// 128-byte-swizzled MN-major tile of W_downT rows (k = neuron, 128 elements
// of d): 16-byte piece c16 of row k; the two 64-element halves of d are
// K2*128 bytes apart, rows k form 1024-byte groups of 8.
__device__ __forceinline__ uint32_t sw128_mn(int k, int c16, int K2) {
  return (uint32_t)((c16 >> 3) * (K2 * 128) + (k >> 3) * 1024 + (k & 7) * 128 + (((c16 & 7) ^ (k & 7)) << 4));
}


}  // namespace tc
}  // namespace sffn
