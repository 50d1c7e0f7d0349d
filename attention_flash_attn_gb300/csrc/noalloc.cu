// noalloc.cu -- attn_fwd_noalloc: the forward pass for callers that cannot allocate device
// memory, with its workspace in a fixed array that lives in the library image.
//
// Callers this is for: plugins hosted by a runtime that owns every device allocation and
// gives them no allocator to call, and deployments whose device-memory budget is fixed up
// front, where a library may not call cudaMalloc on its own.  Such a caller passes its
// inputs and outputs as usual; the scratch the forward needs (the device status word and,
// for packed segments, the segment metadata) comes from g_fwd_scratch below.
//
// The array exists once per GPU context that loads the library and stays resident until the
// process exits.  In host code its name is only a host-side stand-in: the device address is
// looked up with cudaGetSymbolAddress on every call, in the context that is current then --
// a plugin may run in a context of its own, and a context that was destroyed and created
// again holds the array at a new address -- so no address is ever reused across contexts.
// After the first call in a context the lookup is a table read.
#include <cuda_runtime.h>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB
__device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

// Device address of g_fwd_scratch in the current context.
int scratch_in_current_context(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const attn_args *a, void *O, float *LSE, attn_stream_t stream) {
  // attn_fwd's own checks first, in its order, so that both entry points answer a request
  // alike; only then the array's size limit.
  bool empty = false;
  int s = attn::fwd_precheck(a, O, LSE, &empty);
  if (s != ATTN_OK || empty) return s;
  if (attn_fwd_workspace_size(a) > kScratchBytes) return ATTN_ERR_WORKSPACE;
  void *ws = nullptr;
  if ((s = scratch_in_current_context(&ws)) != ATTN_OK) return s;
  // The array keeps the previous call's contents; the status area must start at zero.
  // The segment metadata is rewritten in full by every call that uses it.
  if (cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  return attn_fwd(a, O, LSE, ws, kScratchBytes, stream);
}

extern "C" int attn_noalloc_check_device_status(attn_stream_t stream) {
  void *ws = nullptr;
  const int s = scratch_in_current_context(&ws);
  if (s != ATTN_OK) return s;
  return attn_check_device_status(ws, stream);
}
