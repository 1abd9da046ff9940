// Expert FFN entry point for callers that cannot allocate device memory.
//
// pw_expert_ffn_bitplane needs a scratch buffer from the caller for the fp16
// activations h between the gate/up and the down projections.  Some callers
// cannot provide one at the point where they run the layer: a serving engine
// that has handed all of HBM to its weight pool and KV cache and allows no
// further cudaMalloc, or a host application that only passes pre-allocated
// inputs and outputs into this library.  This variant keeps that scratch in a
// fixed-size array in the library's own device memory instead.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pw_internal.h"

namespace {

// Statically sized scratch: every GPU that loads the library holds it until
// the process exits.  Slots x ffn x 2 bytes of h must fit.
constexpr size_t kNoAllocScratchBytes = 8u << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per
// device; the name is only a host-side stand-in and must never be passed to a kernel).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pw_status pw_expert_ffn_bitplane_noalloc(pw_layer_t layer, const void* x_perm, const int32_t* offsets,
                                                    int T, float* y_perm, void* stream) {
  pw::DevLayer dev;
  int class_mask = 0;
  size_t h_bytes = 0;
  pw_status st = pw::ffn_call_args(layer, x_perm, offsets, T, y_perm, &dev, &class_mask, &h_bytes);
  if (st != PW_OK || T == 0) return st;
  if (h_bytes > kNoAllocScratchBytes) return PW_ERR_OOM;
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return pw::record_cuda_error(e);
  e = pw::launch_moe_ffn(dev, static_cast<const __half*>(x_perm), offsets, T * dev.K, y_perm,
                         static_cast<__half*>(scratch), nullptr, T, nullptr, nullptr, class_mask,
                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PW_OK : pw::record_cuda_error(e);
}
