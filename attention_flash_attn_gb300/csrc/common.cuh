// common.cuh -- definitions shared by every kernel of the library: the kernel parameter
// block, the score modification (scale, bias, tanh soft-cap, visibility) and the device
// status word.  Forward and backward kernels call the same functions so that the
// probabilities they form from a logit are computed identically.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace attn {

// Device status bits (OR-ed into the first word of the workspace).
enum : unsigned {
  kStatusWaitTimeout = 1u,     // a bounded mbarrier / TMEM wait gave up
  kStatusBadCuSeqlens = 2u,    // cu_seqlens not 0-based / non-decreasing / within Sq
  kStatusBadTmemAlloc = 4u,    // tensor-memory allocation returned an unusable address
};

// Everything a kernel needs, passed by value.
struct Params {
  // problem
  int B, Sq, Sk, Hq, Hkv, D, G;   // G = Hq / Hkv
  int causal, window;             // window <= 0: off
  float cap, inv_cap, scale;      // cap == 0: off
  // inputs (element strides)
  const void *q, *k, *v;
  long long q_sb, q_ss, q_sh, k_sb, k_ss, k_sh, v_sb, v_ss, v_sh;
  const void *bias;
  long long bias_sb, bias_sh;
  int bias_B, bias_H;             // extents of the bias's own batch / head dims (1 = broadcast)
  int bias_vec;                   // every bias row starts on a 16-byte boundary (16-byte loads)
  const int *seg_q, *seg_k;       // effective segment ids or null
  const int2 *qrange;             // [B, ceil(Sq/64)]: key range [x, y) of each 64-row query tile
  const int2 *krange;             // [B, ceil(Sk/64)]: query range [x, y) of each 64-key tile
  const int2 *qrun, *krun;        // [B, Sq] / [B, Sk]: each query's key interval [x, y) and each
                                  // key's query interval (mask metadata; null without it)
  const unsigned char *seg_mono;  // [B]: 1 if seg_q and seg_k rows are non-decreasing
  // Tile classes (segment / cu_seqlens calls; null otherwise): per (b, 128-row query tile)
  // {klo, khi, flo, fhi} -- the keys some row of the tile sees lie in [klo, khi), the keys every
  // row sees in [flo, fhi) (empty when flo >= fhi; always empty with unsorted ids).  A key tile
  // inside [flo, fhi) is FULL (no mask needed), one outside [klo, khi) EMPTY, any other PARTIAL.
  // Per (b, 128-key tile) the same over the queries that see its keys.
  const int4 *qtile, *ktile;
  // Longest-first work lists: every (b, 128-row query tile) / (b, 128-key tile) once, as
  // {b, tile}, in descending power-of-two class of visible pairs and, within a class, in the
  // grid's own locality order; null when the call has no segments, more tiles than the sorter
  // takes, or a grid too large to follow a list (the grid's own order then).
  const int2 *qorder, *korder;
  // Varlen with separate key boundaries (B == 1): per token, the causal / window offset of its
  // sequence, end_k(s) - end_q(s) (bottom-right alignment within every sequence); null: the
  // whole matrix's Sk - Sq.
  const int *qoff;                // [Sq]
  const int *koff;                // [Sk]
  const float *sink;              // [Hq] or null
  int off_by_one;                 // one extra column of logit 0 per row (no sink array)
  // Split-KV forward (kv_splits > 1): each split writes its normalised partial output and LSE
  // (without the sink column) here; a merge kernel combines them.
  int kv_splits;
  // Backward grid order without segments: 1 = (batch, kv head) slowest, key tile fastest (long
  // query ranges); 0 = key tile slowest.
  int bwd_group_major;
  float *o_part;                  // [kv_splits, B, Hq, Sq, D]
  float *lse_part;                // [kv_splits, B, Hq, Sq]
  // forward outputs / backward inputs
  void *O;
  float *LSE;
  const void *dO;
  // backward outputs and scratch
  void *dQ, *dK, *dV, *dbias;
  float *dsink;
  float *Dvec;                    // [B, Hq, sq_pad]: D = rowsum(dO * O), 0 past Sq
  float *lse2p;                   // [B, Hq, sq_pad]: LSE * log2(e), +inf past Sq
  uint4 *dsplit;                  // [B, Hq, sq_pad]: -D as bf16 parts (hi, mid, lo, 5 zeros), 0 past Sq; fused tc backward only
  int sq_pad;                     // Sq rounded up to a multiple of 128
  float *dQacc;                   // [B, Sq, Hq, D] fp32 accumulator (tensor-core path)
  float *dbias_acc;               // dense fp32 copy of dbias being accumulated
  float *dsink_part;              // [Hq, n_part]
  int n_part;                     // partial sums per head
  unsigned *status;
};

// The extra softmax column of a row, if any: the learnable sink (logit sink[h]) or the
// off-by-one column (logit 0).  It enters the row's normaliser once and carries no value.
__device__ __forceinline__ bool has_sink_col(const Params &p) { return p.sink != nullptr || p.off_by_one != 0; }
__device__ __forceinline__ float sink_logit(const Params &p, int h) { return p.sink ? p.sink[h] : 0.f; }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Query position on the key axis (bottom-right alignment when Sq != Sk, per sequence when
// the sequences have their own key boundaries).
__device__ __forceinline__ int qpos(const Params &p, int i) { return i + (p.qoff ? p.qoff[i] : p.Sk - p.Sq); }
// The offset that places key j's sequence on the query axis (query i sees key j causally iff
// j <= i + key_off(j) within one sequence).
__device__ __forceinline__ int key_off(const Params &p, int j) { return p.koff ? p.koff[j] : p.Sk - p.Sq; }

// Visibility of key j to query i of batch b: causal, sliding window, segment equality.
__device__ __forceinline__ bool visible(const Params &p, int b, int i, int j) {
  const int ip = qpos(p, i);
  if (p.causal && j > ip) return false;
  if (p.window > 0 && ip - j >= p.window) return false;
  if (p.seg_q && p.seg_q[(size_t)b * p.Sq + i] != p.seg_k[(size_t)b * p.Sk + j]) return false;
  return true;
}

// Accurate soft-cap for the fp32 kernels: t = cap * tanh(u / cap) and the backward factor
// 1 - tanh^2(u / cap).  With e = expm1(-2|y|) in (-1, 0]:
//   tanh|y| = -e / (2 + e),   1 - tanh^2 y = 4 (1 + e) / (2 + e)^2,
// which keeps full relative accuracy both near 0 and deep in saturation.
__device__ __forceinline__ void softcap_accurate(float u, float cap, float inv_cap,
                                                 float &t, float &factor) {
  const float y = u * inv_cap;
  const float e = expm1f(-2.0f * fabsf(y));
  const float d = 2.0f + e;
  const float th = -e / d;
  t = copysignf(cap * th, y);
  factor = 4.0f * (1.0f + e) / (d * d);
}

// Records a device-side error; never traps.
__device__ __forceinline__ void set_status(unsigned *status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace attn
