// Dense fallback for batches whose union of active rows covers most of the
// layer: every row is read once, as two plain GEMMs on the tensor cores
// (cuBLASLt, 16-bit operands, fp32 accumulation and output), with this file's
// kernels between and after them:
//
//   D_up[b][i]  = W_up[i] . x_b   (and D_gate for ReGLU)            GEMM 1
//   a[b][i]     = [i in M_b] ReLU(D_up + b_i)  or  [i in M_b] ReLU(D_gate + b_i) D_up
//   A           = a as a 16-bit high part (rows 0..B-1) and a 16-bit
//                 remainder (rows B..2B-1), so the second product keeps fp32
//                 accuracy                                               (k_dense_act)
//   Y2[r][j]    = sum_i W_down^T[i][j] A[r][i]                           GEMM 2
//   y[b][j]     = Y2[b][j] + Y2[B + b][j]                                (k_dense_combine)
//
// Each token keeps only its own predicted neurons (the token mask M_b is
// applied to a), so the result is the masked FFN of the sparse path; only the
// rows read differ.  When most rows are in the union anyway, one dense pass
// over contiguous rows moves the bytes faster than gathering (the throughput
// paragraph of the sparsity page's section 工程影響: the benefit of sparsity
// decays with the batch; PowerInfer-2 page, 4.1.1: prefill, where sparsity is
// low, runs all neurons as one dense cluster).

#include "kernels.cuh"

namespace sffn {

namespace {

constexpr int kActThreads = 256;

// One thread per (token, neuron); neurons fastest, so the D loads and the A
// stores of a warp are contiguous.
template <typename T>
__global__ void __launch_bounds__(kActThreads)
    k_dense_act(const float* __restrict__ d_up, const float* __restrict__ d_gate, const float* __restrict__ bias,
                const uint32_t* __restrict__ mask, int B, int f, int W, T* __restrict__ A) {
  const int i = blockIdx.x * kActThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (i >= f || b >= B) return;
  const size_t o = (size_t)b * f + i;
  float av = 0.f;
  if ((__ldg(mask + (size_t)b * W + (i >> 5)) >> (i & 31)) & 1u) {
    const float bi = bias != nullptr ? __ldg(bias + i) : 0.f;
    const float u = d_up[o];
    av = d_gate != nullptr ? fmaxf(d_gate[o] + bi, 0.f) * u : fmaxf(u + bi, 0.f);
  }
  const T hi = from_float<T>(av);
  A[o] = hi;
  A[(size_t)(B + b) * f + i] = from_float<T>(av - static_cast<float>(hi));
}

// y[b][j] = Y2[b][j] + Y2[B + b][j], four columns per thread.
__global__ void __launch_bounds__(256) k_dense_combine(const float* __restrict__ y2, int B, int d, float* __restrict__ y) {
  const int q = blockIdx.x * 256 + threadIdx.x;  // float4 index within a row
  const int b = blockIdx.y;
  if (q >= d / 4 || b >= B) return;
  const float4 hi = reinterpret_cast<const float4*>(y2 + (size_t)b * d)[q];
  const float4 lo = reinterpret_cast<const float4*>(y2 + (size_t)(B + b) * d)[q];
  reinterpret_cast<float4*>(y + (size_t)b * d)[q] = make_float4(hi.x + lo.x, hi.y + lo.y, hi.z + lo.z, hi.w + lo.w);
}

template <typename T>
cudaError_t act_launch(const float* d_up, const float* d_gate, const float* bias, const uint32_t* mask, int B, int f,
                       int W, void* A, cudaStream_t s) {
  const dim3 grid((f + kActThreads - 1) / kActThreads, B);
  k_dense_act<T><<<grid, kActThreads, 0, s>>>(d_up, d_gate, bias, mask, B, f, W, static_cast<T*>(A));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_act(int dtype, const float* d_up, const float* d_gate, const float* bias,
                             const uint32_t* mask, int B, int f, int W, void* A, cudaStream_t s) {
  switch (dtype) {
    case kF16: return act_launch<__half>(d_up, d_gate, bias, mask, B, f, W, A, s);
    case kBF16: return act_launch<__nv_bfloat16>(d_up, d_gate, bias, mask, B, f, W, A, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dense_combine(const float* y2, int B, int d, float* y, cudaStream_t s) {
  const dim3 grid((d / 4 + 255) / 256, B);
  k_dense_combine<<<grid, 256, 0, s>>>(y2, B, d, y);
  return cudaGetLastError();
}

}  // namespace sffn
