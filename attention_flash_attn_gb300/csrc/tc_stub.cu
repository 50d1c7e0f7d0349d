// Placeholder until the tcgen05 kernels land: no D is served by the tensor-core path.
#include "common.cuh"
#include "internal.h"
namespace attn {
bool tc_supported(int) { return false; }
cudaError_t tc_forward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t tc_backward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace attn
