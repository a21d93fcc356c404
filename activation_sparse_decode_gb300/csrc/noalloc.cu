// sffn_forward_noalloc: the batch-1 sparse FFN (the single-launch layer
// kernel) with its scratch in a fixed array that lives in the library itself,
// for callers that cannot allocate device memory.
//
// Who cannot allocate: serving loops and embedded runtimes that own all device
// memory up front (a fixed pool handed out by their own allocator) and forbid
// cudaMalloc once running -- cudaMalloc may synchronise the device and
// fragments a pool sized to the byte -- and host programs whose device memory
// belongs to another framework's allocator.  Such a caller still passes its
// token and output buffers; only the kernel's scratch (the workspace header
// with its status word and launch counter, and the tagged slots through which
// the blocks exchange the predictor's hidden layer) comes from here.

#include "../../include/sffn.h"
#include "kernels.cuh"

// Defined in api.cu: the layer's device, the layer kernel on caller-given
// scratch, and the error message of the calling thread.
sffn_status sffn_internal_layer_device(sffn_layer_t layer, int* device);
sffn_status sffn_internal_layer_on_scratch(sffn_layer_t layer, const void* x, float* y, void* scratch,
                                           size_t scratch_bytes, void* stream);
sffn_status sffn_internal_fail(sffn_status status, const char* message);

namespace {

// Scratch of the no-allocation entry point, on every device that loads the
// library, for the life of the process.  Layout (as in a workspace): header
// (256 bytes: status word, launch counter), barrier release flags (128 bytes
// per block), the tagged hidden-layer slots (128 bytes per predictor rank
// row).  Shared by every call.
constexpr size_t kScratchBytes = 256 * 1024;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device: in host code the
// array's name is only a stand-in, never a device address.  Looked up on
// every call (a host-side table lookup once the module is loaded), so that a
// context torn down and created again is never handed a stale address.  The
// first lookup on a device loads the library's kernels there, which is why
// the first call on a device must come before any stream capture.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" sffn_status sffn_forward_noalloc(sffn_layer_t layer, const void* x, float* y, void* stream) {
  int device = -1;
  const sffn_status st = sffn_internal_layer_device(layer, &device);
  if (st != SFFN_OK) return st;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return sffn_internal_fail(SFFN_ERR_CUDA, "cudaGetDevice failed");
  if (cur != device)
    return sffn_internal_fail(SFFN_ERR_INVALID_ARG, "the layer was created on another device than the current one");
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess)
    return sffn_internal_fail(SFFN_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
  return sffn_internal_layer_on_scratch(layer, x, y, scratch, kScratchBytes, stream);
}

extern "C" sffn_status sffn_noalloc_read_status(int32_t* status, void* stream) {
  if (status == nullptr) return sffn_internal_fail(SFFN_ERR_INVALID_ARG, "status is NULL");
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess)
    return sffn_internal_fail(SFFN_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
  // the first two header words: the sticky status and where it was raised
  uint32_t words[2] = {0u, 0u};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(words, scratch, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return sffn_internal_fail(SFFN_ERR_CUDA, "reading the status word failed");
  *status = (int32_t)words[0];
  if (words[0] != 0u &&
      (cudaMemsetAsync(scratch, 0, sizeof(words), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess))
    return sffn_internal_fail(SFFN_ERR_CUDA, "clearing the status word failed");
  return SFFN_OK;
}
