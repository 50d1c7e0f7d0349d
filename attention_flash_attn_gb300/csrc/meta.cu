// meta.cu -- mask metadata for packed segments (segment ids or cu_seqlens).
//
// One kernel, one warp per 128-row tile of either axis: it turns cu_seqlens into segment ids
// when given (with separate key boundaries, ids per axis and each token's per-sequence
// bottom-right offset), decides whether each batch row's ids are non-decreasing, writes for
// every 64-row query tile the key range [lo, hi) its rows can see and for every 64-key tile
// the query range that can see it (intersected with the causal and window bounds), and for
// every 128-row query tile and 128-key tile (the CTAs of the tensor-core kernels) its tile
// class and its visible pairs.  A second kernel sorts the tiles into longest-first work lists,
// which the tensor-core grids follow (MaxText commit message quoted on tokamax PR #1121: packed
// rows with segments of very different lengths, run starts per row).
// With non-decreasing ids a segment is one contiguous run: read straight from the boundaries
// with cu_seqlens, found by binary search in given ids; with arbitrary ids the ranges fall back
// to the causal/window bounds alone and the kernels test id equality pair by pair.  An empty
// range is stored as {n, 0} so that the union of two tile ranges (min of lo, max of hi)
// ignores it.
#include <algorithm>
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

// One pass.  Grid: x over the 128-row tiles of one axis (eight per block, one per warp), y the
// batch row, z the axis (0: query tiles, 1: key tiles); 256 threads.
//  (1) Sortedness, decided alike by every block: with cu_seqlens, whether the boundaries pass
//      their checks (they then give non-decreasing ids by construction; a failed check is
//      recorded by block (0, 0, 0) and the ids are treated as unsorted, so that the kernels
//      compare ids pair by pair and every access stays inside its array); with given ids,
//      whether both axes' ids of the batch row are non-decreasing.  Block (0, b, 0) stores it.
//  (2) With cu_seqlens, each warp writes the sequence ids of its tile's rows (with
//      cu_seqlens_k also their per-sequence bottom-right offsets end_k(s) - end_q(s)).
//  (3) Each warp: every row's visible interval on the other axis, stored per token (the
//      kernels read it instead of searching), its tile's class and work, and the 64-row ranges
//      of its two halves: every
//      row's visible interval (causal / window bounds at its offset; with sorted ids, its
//      segment's run on the other axis -- read from the boundaries (sequence s spans
//      [cu[s], cu[s + 1]), tokens at or past cu[nseq] forming sequence nseq), or found by binary
//      search in the other axis's ids, kept in shared memory when they fit), their union and
//      intersection, and the sum of their lengths: the tile's visible pairs per head (an upper
//      bound with unsorted ids, where the kernels test pairs one by one and no tile is FULL).
// A standalone build (clear_status) first clears the buffer's own status area, in block
// (0, 0, 0) before anything can be recorded there.
constexpr int kCuSmem = 4096;        // boundaries kept in shared memory at most, per axis
constexpr int kMetaSmemIds = 49152;  // given ids of the other axis in shared memory (192 KiB) at most
__global__ void __launch_bounds__(256) meta_kernel(Params p, const int *cu, const int *cu_k, int nseq, MetaOut o,
                                                   int clear_status) {
  extern __shared__ int sm[];
  const int b = blockIdx.y;
  const bool qside = blockIdx.z == 0;
  const bool first = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  if (clear_status) {  // uniform over the grid
    if (first && threadIdx.x < 64) p.status[threadIdx.x] = 0u;
    __syncthreads();
  }
  const int n_rows = qside ? p.Sq : p.Sk, n_other = qside ? p.Sk : p.Sq;
  const int *cq = cu, *ck = cu_k ? cu_k : cu;  // boundaries of the query and key axes
  const int *own = nullptr, *other = nullptr;
  bool sorted;
  if (cu) {
    if (nseq + 1 <= kCuSmem) {
      for (int x = threadIdx.x; x <= nseq; x += blockDim.x) {
        sm[x] = cu[x];
        if (cu_k) sm[kCuSmem + x] = cu_k[x];
      }
      __syncthreads();
      cq = sm;
      ck = cu_k ? sm + kCuSmem : sm;
    }
    const int bad = __syncthreads_or(bad_bounds(cq, nseq, p.Sq) || (cu_k && bad_bounds(ck, nseq, p.Sk)));
    if (first && threadIdx.x == 0 && bad) set_status(p.status, kStatusBadCuSeqlens);
    sorted = !bad;
  } else {
    own = (qside ? p.seg_q : p.seg_k) + (size_t)b * n_rows;
    other = (qside ? p.seg_k : p.seg_q) + (size_t)b * n_other;
    const bool same = own == other && n_rows == n_other;  // one id array for both axes
    if (n_other <= kMetaSmemIds) {
#pragma unroll 4
      for (int x = threadIdx.x; x < n_other; x += blockDim.x) sm[x] = other[x];
      __syncthreads();
      other = sm;
    }
    int ok = 1;
#pragma unroll 4
    for (int x = threadIdx.x; x + 1 < n_other; x += blockDim.x) ok &= other[x] <= other[x + 1];
    if (!same) {
#pragma unroll 4
      for (int x = threadIdx.x; x + 1 < n_rows; x += blockDim.x) ok &= own[x] <= own[x + 1];
    }
    sorted = __syncthreads_and(ok);
  }
  if (blockIdx.x == 0 && qside && threadIdx.x == 0) o.mono[b] = (unsigned char)sorted;

  const int *cu_own = qside ? cq : ck, *cu_oth = qside ? ck : cq;
  const bool per_seq = cu && cu_k;
  const int off = p.Sk - p.Sq;
  const int n64 = (n_rows + 63) / 64;
  const int lane = threadIdx.x & 31;
  const int n128 = (n_rows + 127) / 128;
  const int tt = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tt < n128) {
    int lo_min = INT_MAX, hi_max = INT_MIN, lo_max = INT_MIN, hi_min = INT_MAX;
    int h_lo[2] = {INT_MAX, INT_MAX}, h_hi[2] = {INT_MIN, INT_MIN};  // per 64-row half
    long long work = 0;
    for (int r = tt * 128 + lane; r < min(tt * 128 + 128, n_rows); r += 32) {
      int id, so = off;
      if (cu) {
        id = seq_of(cu_own, nseq, r);
        if (per_seq) so = seq_end(ck, nseq, p.Sk, id) - seq_end(cq, nseq, p.Sq, id);
        if (qside) {
          o.seg_q[r] = id;
          if (per_seq) o.qoff[r] = so;
        } else if (per_seq) {
          o.seg_k[r] = id;
          o.koff[r] = so;
        }
      } else {
        id = own[r];
      }
      int lo, hi;
      if (qside) {
        const int ip = r + so;  // position on the key axis
        lo = p.window > 0 ? ip - p.window + 1 : 0;
        hi = p.causal ? ip + 1 : p.Sk;
      } else {
        const int kp = r - so;  // position on the query axis
        lo = p.causal ? kp : 0;
        hi = p.window > 0 ? kp + p.window : p.Sq;
      }
      if (sorted) {
        if (cu) {  // checked boundaries: id in [0, nseq], non-decreasing, within n_other
          lo = max(lo, cu_oth[id]);
          hi = min(hi, id < nseq ? cu_oth[id + 1] : n_other);
        } else {
          lo = max(lo, lower_bound_i(other, n_other, id));
          hi = min(hi, upper_bound_i(other, n_other, id));
        }
      }
      lo = max(lo, 0);
      hi = min(hi, n_other);
      (qside ? o.qrun : o.krun)[(size_t)b * n_rows + r] = make_int2(lo, hi);
      lo_max = max(lo_max, lo);
      hi_min = min(hi_min, hi);
      if (lo < hi) {
        lo_min = min(lo_min, lo);
        hi_max = max(hi_max, hi);
        work += hi - lo;
        const int hf = (r >> 6) & 1;
        h_lo[hf] = min(h_lo[hf], lo);
        h_hi[hf] = max(h_hi[hf], hi);
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      h_lo[hf] = __reduce_min_sync(0xffffffffu, h_lo[hf]);
      h_hi[hf] = __reduce_max_sync(0xffffffffu, h_hi[hf]);
      const int t64 = 2 * tt + hf;
      if (lane == 0 && t64 < n64)
        (qside ? o.qrange : o.krange)[(size_t)b * n64 + t64] =
            h_lo[hf] < h_hi[hf] ? make_int2(h_lo[hf], h_hi[hf]) : make_int2(n_other, 0);
    }
    lo_min = __reduce_min_sync(0xffffffffu, lo_min);
    hi_max = __reduce_max_sync(0xffffffffu, hi_max);
    lo_max = __reduce_max_sync(0xffffffffu, lo_max);
    hi_min = __reduce_min_sync(0xffffffffu, hi_min);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) work += __shfl_xor_sync(0xffffffffu, work, x);
    if (lane == 0) {
      // A key tile that runs past Sk has no FULL query steps: the backward kernel computes P
      // for its missing keys too, and only the mask keeps them out (as the kernel's own
      // per-key intersection would, those keys seeing nothing).  Query rows past Sq are never
      // stored, so a query tile's class ignores them.
      const bool full_ok = sorted && (qside || tt * 128 + 128 <= p.Sk);
      const int4 c = lo_min < hi_max ? make_int4(lo_min, hi_max, full_ok ? lo_max : 0, full_ok ? hi_min : 0)
                                     : make_int4(n_other, 0, 0, 0);
      (qside ? o.qtile : o.ktile)[(size_t)b * n128 + tt] = c;
      (qside ? o.qwork : o.kwork)[(size_t)b * n128 + tt] = work;
    }
  }
}

// Longest-first work list of n tiles (n <= kSortMax): block 0 sorts the query tiles, block 1
// the key tiles.  Tiles are ranked by the power of two of their visible pairs, heaviest class
// first; within a class they keep the grid's locality order (query tiles latest first, key
// tiles earliest first, the batch row fastest), so that tiles of one segment that run together
// still share their key / query tiles in L2 -- ranking by exact work scatters them over rows
// and segments and measured 10-13 % slower on packed rows.  A bitonic sort in shared memory of
// the keys class * 2^20 + (2^20 - 1 - locality rank), descending; entry e of the list is
// {b, tile} of the e-th tile.
constexpr int kSortMax = 4096;
__global__ void __launch_bounds__(1024) work_order_kernel(const long long *qwork, int nq, int nqt, int2 *qorder,
                                                          const long long *kwork, int nk, int nkt, int2 *korder) {
  __shared__ unsigned long long key[kSortMax];
  const bool qside = blockIdx.x == 0;
  const long long *work = qside ? qwork : kwork;
  const int n = qside ? nq : nk, per_row = qside ? nqt : nkt, nb = n / max(per_row, 1);
  int2 *order = qside ? qorder : korder;
  if (n <= 0 || n > kSortMax) return;
  int m = 1;
  while (m < n) m <<= 1;
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    unsigned long long kv = 0ull;
    if (i < n) {
      const int b = i / per_row, t = i % per_row;
      const int rank = (qside ? per_row - 1 - t : t) * nb + b;  // the grid's own order
      const unsigned long long cls = 64 - __clzll((unsigned long long)work[i] + 1);
      kv = (cls << 20) | (unsigned long long)(0xFFFFF - rank);
    }
    key[i] = kv;
  }
  __syncthreads();
  for (int size = 2; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const int jx = i ^ stride;
        if (jx > i) {
          const bool desc = (i & size) == 0;  // descending runs first: the whole array ends descending
          const unsigned long long a = key[i], c = key[jx];
          if (desc ? a < c : a > c) {
            key[i] = c;
            key[jx] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int rank = 0xFFFFF - (int)(key[e] & 0xFFFFFull);
    const int b = rank % nb, r = rank / nb;
    order[e] = make_int2(b, qside ? per_row - 1 - r : r);
  }
}

}  // namespace

cudaError_t launch_mask_meta(const Params &p, const int *cu_seqlens, const int *cu_seqlens_k, int nseq,
                             const MetaOut &o, cudaStream_t st) {
  // blocks along x: one warp per 128-row tile of the longer axis, eight per block
  const long long blocks = ((long long)(std::max(p.Sq, p.Sk) + 127) / 128 + 7) / 8;
  if (blocks > 0x7fffffffLL || p.B > 65535) return cudaErrorInvalidValue;
  size_t smem = 0;
  if (cu_seqlens) {
    if (nseq + 1 <= kCuSmem) smem = 2 * kCuSmem * sizeof(int);
  } else {
    // The blocks of each axis keep the other axis's ids in shared memory when they fit; the
    // launch holds the larger of the two that do (with Sq != Sk one axis may fit alone).
    int n_ids = 0;
    if (p.Sk <= kMetaSmemIds) n_ids = std::max(n_ids, p.Sk);
    if (p.Sq <= kMetaSmemIds) n_ids = std::max(n_ids, p.Sq);
    smem = (size_t)n_ids * sizeof(int);
  }
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  meta_kernel<<<dim3((unsigned)std::max(blocks, 1LL), (unsigned)p.B, 2), 256, smem, st>>>(p, cu_seqlens, cu_seqlens_k,
                                                                                        nseq, o, o.clear_status);
  e = counted(cudaGetLastError());
  if (e != cudaSuccess || !o.qorder) return e;
  const int nqt = (p.Sq + 127) / 128, nkt = (p.Sk + 127) / 128;
  work_order_kernel<<<2, 1024, 0, st>>>(o.qwork, p.B * nqt, nqt, o.qorder, o.kwork, p.B * nkt, nkt, o.korder);
  return counted(cudaGetLastError());
}

int work_order_max_tiles() { return kSortMax; }

int device_sm_count() {
  static int sms[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    sms[dev] = n;
  }
  return sms[dev];
}

bool follow_work_list(long long nblk) { return nblk <= 4LL * device_sm_count(); }

}  // namespace attn
