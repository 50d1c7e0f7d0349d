// meta.cu -- mask metadata for packed segments (segment ids or cu_seqlens).
//
// One block per batch row.  It (1) turns cu_seqlens into segment ids when given (with
// separate key boundaries, ids per axis and each token's per-sequence bottom-right offset),
// (2) checks whether the row's query and key ids are non-decreasing, and (3) for every
// 64-row query tile writes the key range [lo, hi) its rows can see, and for every 64-key
// tile the query range that can see it, intersected with the causal and window bounds.
// With non-decreasing ids a segment is one contiguous run, found by binary search; with
// arbitrary ids the ranges fall back to the causal/window bounds alone and the kernels
// test id equality pair by pair.  An empty range is stored as {n, 0} so that the union of
// two tile ranges (min of lo, max of hi) ignores it.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

// First index in a[0..n) with a[idx] >= x (a non-decreasing).
__device__ int lower_bound_i(const int *a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}
// First index in a[0..n) with a[idx] > x.
__device__ int upper_bound_i(const int *a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Sequence of token t under boundaries cu[0..nseq]: s with cu[s] <= t < cu[s + 1]; tokens at or
// past cu[nseq] form sequence nseq.
__device__ __forceinline__ int seq_of(const int *cu, int nseq, int t) {
  const int s = upper_bound_i(cu, nseq + 1, t) - 1;
  return s < 0 ? 0 : s;
}
// End (exclusive) of sequence s on an axis of n tokens.
__device__ __forceinline__ int seq_end(const int *cu, int nseq, int n, int s) { return s < nseq ? cu[s + 1] : n; }

__device__ __forceinline__ bool bad_bounds(const int *cu, int nseq, int n) {
  bool bad = false;
  if (threadIdx.x == 0) bad = cu[0] != 0 || cu[nseq] > n;
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) bad |= cu[s] > cu[s + 1];
  return bad;
}

__global__ void __launch_bounds__(1024) mask_meta_kernel(Params p, const int *cu, const int *cu_k, int nseq,
                                                         int *seg_out, int *segk_out, int *qoff_out,
                                                         int *koff_out, int2 *qrange, int2 *krange,
                                                         unsigned char *mono) {
  const int b = blockIdx.x;
  const int *sq, *sk;
  if (cu && cu_k) {
    // B == 1, separate query and key boundaries: ids per axis, and per token the bottom-right
    // offset end_k(s) - end_q(s) of its sequence.
    if (bad_bounds(cu, nseq, p.Sq) || bad_bounds(cu_k, nseq, p.Sk)) set_status(p.status, kStatusBadCuSeqlens);
    for (int t = threadIdx.x; t < p.Sq; t += blockDim.x) {
      const int s = seq_of(cu, nseq, t);
      seg_out[t] = s;
      qoff_out[t] = seq_end(cu_k, nseq, p.Sk, s) - seq_end(cu, nseq, p.Sq, s);
    }
    for (int t = threadIdx.x; t < p.Sk; t += blockDim.x) {
      const int s = seq_of(cu_k, nseq, t);
      segk_out[t] = s;
      koff_out[t] = seq_end(cu_k, nseq, p.Sk, s) - seq_end(cu, nseq, p.Sq, s);
    }
    __syncthreads();
    sq = seg_out;
    sk = segk_out;
  } else if (cu) {
    // B == 1 and Sq == Sk: one id array serves queries and keys.
    if (bad_bounds(cu, nseq, p.Sq)) set_status(p.status, kStatusBadCuSeqlens);
    for (int t = threadIdx.x; t < p.Sq; t += blockDim.x) seg_out[t] = seq_of(cu, nseq, t);
    __syncthreads();
    sq = sk = seg_out;
  } else {
    sq = p.seg_q + (size_t)b * p.Sq;
    sk = p.seg_k + (size_t)b * p.Sk;
  }
  int ok = 1;
  for (int i = threadIdx.x; i + 1 < p.Sq; i += blockDim.x) ok &= sq[i] <= sq[i + 1];
  for (int j = threadIdx.x; j + 1 < p.Sk; j += blockDim.x) ok &= sk[j] <= sk[j + 1];
  const int sorted = __syncthreads_and(ok);
  if (threadIdx.x == 0) mono[b] = (unsigned char)sorted;

  // Causal / window bounds of a tile: the union of its rows' intervals.  With one offset for
  // the whole matrix the first / last row decide them; with per-sequence offsets every row
  // of the tile is visited.
  const bool per_seq = cu && cu_k;
  const int off = p.Sk - p.Sq;
  const int nqt = (p.Sq + 63) / 64, nkt = (p.Sk + 63) / 64;
  for (int t = threadIdx.x; t < nqt; t += blockDim.x) {
    const int i0 = t * 64, i1 = min(i0 + 64, p.Sq) - 1;
    int lo = 0, hi = p.Sk;
    if (sorted) {
      lo = lower_bound_i(sk, p.Sk, sq[i0]);
      hi = upper_bound_i(sk, p.Sk, sq[i1]);
    }
    int cl = i0 + off - p.window + 1, ch = i1 + off + 1;  // window floor, causal ceiling
    if (per_seq) {
      cl = INT_MAX;
      ch = INT_MIN;
      for (int i = i0; i <= i1; ++i) {
        cl = min(cl, i + qoff_out[i] - p.window + 1);
        ch = max(ch, i + qoff_out[i] + 1);
      }
    }
    if (p.causal) hi = min(hi, ch);
    if (p.window > 0) lo = max(lo, cl);
    lo = max(lo, 0);
    hi = min(hi, p.Sk);
    qrange[(size_t)b * nqt + t] = lo < hi ? make_int2(lo, hi) : make_int2(p.Sk, 0);
  }
  for (int t = threadIdx.x; t < nkt; t += blockDim.x) {
    const int j0 = t * 64, j1 = min(j0 + 64, p.Sk) - 1;
    int lo = 0, hi = p.Sq;
    if (sorted) {
      lo = lower_bound_i(sq, p.Sq, sk[j0]);
      hi = upper_bound_i(sq, p.Sq, sk[j1]);
    }
    int cl = j0 - off, ch = j1 - off + p.window;  // causal floor, window ceiling
    if (per_seq) {
      cl = INT_MAX;
      ch = INT_MIN;
      for (int j = j0; j <= j1; ++j) {
        cl = min(cl, j - koff_out[j]);
        ch = max(ch, j - koff_out[j] + p.window);
      }
    }
    if (p.causal) lo = max(lo, cl);
    if (p.window > 0) hi = min(hi, ch);
    lo = max(lo, 0);
    hi = min(hi, p.Sq);
    krange[(size_t)b * nkt + t] = lo < hi ? make_int2(lo, hi) : make_int2(p.Sq, 0);
  }
}

}  // namespace

cudaError_t launch_mask_meta(const Params &p, const int *cu_seqlens, const int *cu_seqlens_k, int nseq,
                             int *seg_q_out, int *seg_k_out, int *qoff_out, int *koff_out, int2 *qrange,
                             int2 *krange, unsigned char *mono, cudaStream_t st) {
  mask_meta_kernel<<<p.B, 1024, 0, st>>>(p, cu_seqlens, cu_seqlens_k, nseq, seg_q_out, seg_k_out, qoff_out,
                                         koff_out, qrange, krange, mono);
  return counted(cudaGetLastError());
}

}  // namespace attn
