// noalloc.cu -- attn_fwd_noalloc: the forward pass for callers that cannot allocate device
// memory, with its workspace in a fixed array that lives in the library image.
//
// Callers this is for: plugins hosted by a runtime that owns every device allocation and
// gives them no allocator to call, and deployments whose device-memory budget is fixed up
// front, where a library may not call cudaMalloc on its own.  Such a caller passes its
// inputs and outputs as usual; the scratch the forward needs (the device status word and,
// for packed segments, the segment metadata) comes from g_fwd_scratch below.
//
// The array exists once per GPU that loads the library and stays resident until the process
// exits.  In host code its name is only a host-side stand-in: the device address is looked
// up with cudaGetSymbolAddress, once per device, with that device current.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn_gb300.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB
__device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void *g_dev_ptr[kMaxDevices];

// Device address of g_fwd_scratch on the current device (looked up once per device).
int scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_dev_ptr[dev] = p;
  }
  *out = g_dev_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const attn_args *a, void *O, float *LSE, attn_stream_t stream) {
  const size_t need = attn_fwd_workspace_size(a);
  if (need == 0) return attn_fwd(a, O, LSE, nullptr, 0, stream);  // reports the validation error
  if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;
  void *ws = nullptr;
  int s = scratch_for_current_device(&ws);
  if (s != ATTN_OK) return s;
  // The array keeps the previous call's contents; the status word must start at zero.
  // The segment metadata is rewritten in full by every call that uses it.
  if (cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  return attn_fwd(a, O, LSE, ws, kScratchBytes, stream);
}
