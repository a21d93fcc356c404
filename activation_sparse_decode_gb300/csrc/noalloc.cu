// sffn_forward_noalloc: the batch-1 sparse FFN (the single-launch layer
// kernel) with its scratch in a fixed array that lives in the library itself,
// for callers that cannot allocate device memory.
//
// Who cannot allocate: serving loops and embedded runtimes that own all device
// memory up front (a fixed pool handed out by their own allocator) and forbid
// cudaMalloc once running -- cudaMalloc may synchronise the device and
// fragments a pool sized to the byte -- and host programs whose device memory
// belongs to another framework's allocator.  Such a caller still passes its
// token and output buffers; only the kernel's scratch (barrier words, the
// predictor's split-K partial sums) comes from here.

#include <mutex>

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
// (256 bytes), barrier release flags (128 bytes per block), predictor partial
// sums.  Shared by every call.
constexpr size_t kScratchBytes = 256 * 1024;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `device`, which must be current: in
// host code the array's name is only a stand-in, never a device address.  Set
// up once per device, on the first call there.
cudaError_t scratch_address(int device, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
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
  if (device < 0 || device >= kMaxDevices) return sffn_internal_fail(SFFN_ERR_UNSUPPORTED, "device index above 63");
  void* scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess)
    return sffn_internal_fail(SFFN_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
  return sffn_internal_layer_on_scratch(layer, x, y, scratch, kScratchBytes, stream);
}
