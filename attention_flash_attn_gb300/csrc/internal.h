// internal.h -- host-side declarations shared by the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "../../include/attn_gb300.h"

namespace attn {

// attn_fwd's checks that come before any workspace is looked at: argument validation, then
// (when there is something to compute) the outputs.  Returns an attn_status; *empty is set
// when B == 0 or Sq == 0 (nothing to compute, ATTN_OK).
int fwd_precheck(const attn_args *a, const void *O, const float *LSE, bool *empty);

struct Params;

enum { kBF16 = 1, kF32 = 2 };

// Kernels launched by this library in this process (see attn_launch_counter).
extern std::atomic<unsigned long long> g_launches;
inline cudaError_t counted(cudaError_t e, int n = 1) {
  if (e == cudaSuccess) g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed);
  return e;
}

// Mask metadata (segments / cu_seqlens): effective segment ids, per-batch monotonicity,
// 64-granular tile ranges, 128-granular tile classes and work, and the longest-first work
// lists.  seg_q is only written when cu_seqlens is given (then B == 1); seg_k, qoff and koff
// only when cu_seqlens_k is given as well; qorder / korder only when non-null (at most
// work_order_max_tiles() tiles per axis).
struct MetaOut {
  int *seg_q, *seg_k, *qoff, *koff;
  int2 *qrange, *krange;
  int2 *qrun, *krun;  // per-token visible intervals on the other axis
  unsigned char *mono;
  int4 *qtile, *ktile;
  long long *qwork, *kwork;
  int2 *qorder, *korder;
  int clear_status;  // a standalone build: clear the buffer's own status area first
};
cudaError_t launch_mask_meta(const Params &p, const int *cu_seqlens, const int *cu_seqlens_k, int nseq,
                             const MetaOut &o, cudaStream_t st);
int work_order_max_tiles();
// Whether a tensor-core grid of nblk one-CTA-per-SM blocks follows the work list: only when it
// spans at most four waves on the current device.  With few waves the tail decides the time and
// longest-first wins (chunked prefill forward +23 %); with many, the grid's own order keeps
// neighbouring tiles of a segment -- which read the same key or query tiles -- running together
// in L2, and measured 5-13 % faster (packed rows, forward and backward; chunked prefill
// backward).
bool follow_work_list(long long nblk);
// Streaming multiprocessors of the current device (cached per device; 1 if the query fails).
int device_sm_count();

// fp32 FFMA kernels (any dtype; used for fp32 inputs and calls with a bias).
cudaError_t simt_forward(const Params &p, int dtype, cudaStream_t st);
cudaError_t simt_backward(const Params &p, int dtype, cudaStream_t st);

// Backward preprocess: D = rowsum(dO * O), per-block dsink partials, zero the fp32 dQ
// accumulator when one is used.
cudaError_t launch_bwd_pre(const Params &p, int dtype, bool zero_dqacc, cudaStream_t st);
int bwd_pre_rows(int B, int Sq, int Hq);      // query positions per preprocess block
int bwd_pre_partials(int B, int Sq, int Hq);  // partial sums per head the preprocess writes
int bwd_pre_partials_max(int B, int Sq);      // ... at most, whatever the block size (workspace)

// Backward epilogue: dQ accumulator -> dQ (when used), dsink reduction, dbias conversion.
cudaError_t launch_bwd_post(const Params &p, int dtype, bool convert_dq, size_t dbias_elems,
                            cudaStream_t st);

// Split-KV forward: merges the kv_splits partial outputs / LSEs into O and LSE, adding the
// sink (or off-by-one) column once.
cudaError_t launch_splitkv_merge(const Params &p, cudaStream_t st);

// tcgen05 tensor-core kernels (bf16, D in {64, 128, 256}).
bool tc_supported(int D);      // forward
bool tc_bwd_supported(int D);  // backward
bool tc_bwd_fused(int D);      // the backward's one-pass form (it reads -D split into bf16 parts)
cudaError_t tc_forward(const Params &p, cudaStream_t st);
cudaError_t tc_backward(const Params &p, cudaStream_t st);

// Head dims 320-512 backward on the tensor cores: a scores kernel writing P and dU into scratch
// [B, Hq, Sq_pad, Sk_pad] (two bf16 planes, wide_bwd_scratch_bytes) and three GEMMs for dV,
// dK, dQ.  Needs LSE * log2(e) and D from the preprocess; writes dQ directly.
size_t wide_bwd_scratch_bytes(int B, int Hq, int Sq, int Sk);
cudaError_t wide_backward(const Params &p, void *scratch, cudaStream_t st);

}  // namespace attn
