// selftest.cu -- attn_selftest_wait_expiry: runs the kernels' bounded-wait failure path on
// purpose, so that it can be checked on the device without any fault.
//
// The kernels never spin forever: every mbarrier wait gives up after a time limit, records
// what it was waiting for in the workspace's status area and lets its CTA wind down, and a
// later kernel that sees the status bit returns at once (TransformerEngine PR #3391, "What
// changed": fail closed rather than silently produce a wrong result).  A correct kernel never
// reaches that path, so this entry point builds the one situation that does: a wait on an
// mbarrier that nothing will ever complete.  The waits are the production ones (mbar_wait),
// with a short limit for the first and the kernels' own limit for the others.
//
// Grid: two CTAs of two warps; lane 0 of a warp does the waiting.
//   CTA 0, warp 0: waits on barrier A (phase 0) with the caller's limit; gives up and
//                  records the first timeout (status words 1-6: marker, barrier, parity,
//                  CTA, thread).
//   CTA 0, warp 1: waits on barrier B with the kernels' limit; gives up as soon as it sees
//                  the status bit and, being in the CTA that recorded the timeout, leaves its
//                  own barrier and parity in words 10 and 11 (words 8 + 2w, 9 + 2w for warp w).
//   CTA 1, warp 0: waits on its own barrier with the kernels' limit and gives up on the
//                  status bit without recording anything (another CTA recorded the timeout).
// Words 48 and 49 receive the shared-memory addresses of A and B, for the caller to compare.
#include <stdint.h>

#include "../../include/attn_gb300.h"
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64) wait_expiry_selftest_kernel(unsigned *status, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bars[2];
  const uint32_t bar_a = smem_u32(&bars[0]), bar_b = smem_u32(&bars[1]);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    mbar_init(bar_b, 1);
    fence_barrier_init();
    if (blockIdx.x == 0) {
      status[48] = bar_a;
      status[49] = bar_b;
    }
  }
  __syncthreads();
  // Warp 0 of CTA 0 gives up first (short limit); the others follow through the status bit.
  if ((threadIdx.x & 31) == 0) {
    if (blockIdx.x == 0)
      (void)mbar_wait(warp == 0 ? bar_a : bar_b, 0, status, warp == 0 ? (uint64_t)limit_ns : kWaitLimitNs);
    else if (warp == 0)
      (void)mbar_wait(bar_a, 0, status, kWaitLimitNs);
  }
  __syncwarp();
  __syncthreads();
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_selftest_wait_expiry(void *ws, size_t ws_bytes, uint64_t limit_ns, attn_stream_t stream) {
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) % 256) != 0) return ATTN_ERR_WORKSPACE;
  if (limit_ns < 1000ull || limit_ns > tc::kWaitLimitNs) return ATTN_ERR_INVALID;
  wait_expiry_selftest_kernel<<<2, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<unsigned *>(ws),
                                                                                     limit_ns);
  return counted(cudaGetLastError()) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
