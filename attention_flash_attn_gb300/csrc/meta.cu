// meta.cu -- mask metadata for packed segments (segment ids or cu_seqlens).
//
// One block per batch row.  It (1) turns cu_seqlens into segment ids when given,
// (2) checks whether the row's query and key ids are non-decreasing, and (3) for every
// 64-row query tile writes the key range [lo, hi) its rows can see, and for every 64-key
// tile the query range that can see it, intersected with the causal and window bounds.
// With non-decreasing ids a segment is one contiguous run, found by binary search; with
// arbitrary ids the ranges fall back to the causal/window bounds alone and the kernels
// test id equality pair by pair.  An empty range is stored as {n, 0} so that the union of
// two tile ranges (min of lo, max of hi) ignores it.
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

__global__ void __launch_bounds__(1024) mask_meta_kernel(Params p, const int *cu, int nseq,
                                                         int *seg_out, int2 *qrange,
                                                         int2 *krange, unsigned char *mono) {
  const int b = blockIdx.x;
  const int *sq, *sk;
  if (cu) {
    // B == 1 and Sq == Sk: one id array serves queries and keys.
    bool bad = false;
    if (threadIdx.x == 0) bad = cu[0] != 0 || cu[nseq] > p.Sq;
    for (int s = threadIdx.x; s < nseq; s += blockDim.x) bad |= cu[s] > cu[s + 1];
    if (bad) set_status(p.status, kStatusBadCuSeqlens);
    for (int t = threadIdx.x; t < p.Sq; t += blockDim.x) {
      // sequence s with cu[s] <= t < cu[s+1]; tokens past cu[nseq] form sequence nseq
      int s = upper_bound_i(cu, nseq + 1, t) - 1;
      seg_out[t] = s < 0 ? 0 : s;
    }
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

  const int off = p.Sk - p.Sq;
  const int nqt = (p.Sq + 63) / 64, nkt = (p.Sk + 63) / 64;
  for (int t = threadIdx.x; t < nqt; t += blockDim.x) {
    const int i0 = t * 64, i1 = min(i0 + 64, p.Sq) - 1;
    int lo = 0, hi = p.Sk;
    if (sorted) {
      lo = lower_bound_i(sk, p.Sk, sq[i0]);
      hi = upper_bound_i(sk, p.Sk, sq[i1]);
    }
    if (p.causal) hi = min(hi, i1 + off + 1);
    if (p.window > 0) lo = max(lo, i0 + off - p.window + 1);
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
    if (p.causal) lo = max(lo, j0 - off);
    if (p.window > 0) hi = min(hi, j1 - off + p.window);
    lo = max(lo, 0);
    hi = min(hi, p.Sq);
    krange[(size_t)b * nkt + t] = lo < hi ? make_int2(lo, hi) : make_int2(p.Sq, 0);
  }
}

}  // namespace

cudaError_t launch_mask_meta(const Params &p, const int *cu_seqlens, int nseq, int *seg_q_out,
                             int *seg_k_out, int2 *qrange, int2 *krange, unsigned char *mono,
                             cudaStream_t st) {
  (void)seg_k_out;  // with cu_seqlens the key ids are the query ids
  mask_meta_kernel<<<p.B, 1024, 0, st>>>(p, cu_seqlens, nseq, seg_q_out, qrange, krange, mono);
  return counted(cudaGetLastError());
}

}  // namespace attn
