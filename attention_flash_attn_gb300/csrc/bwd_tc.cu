// bwd_tc.cu -- tcgen05 tensor-core backward (bf16).  Not yet built: the FFMA backward
// serves every call until it lands.
#include "common.cuh"
#include "internal.h"
namespace attn {
bool tc_bwd_supported(int) { return false; }
cudaError_t tc_backward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace attn
