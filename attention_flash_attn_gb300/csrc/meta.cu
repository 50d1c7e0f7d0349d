// meta.cu -- mask metadata for packed segments (segment ids or cu_seqlens).
//
// A row pass (1) turns cu_seqlens into segment ids when given (with separate key boundaries,
// ids per axis and each token's per-sequence bottom-right offset), spread over as many blocks
// as the tokens need, and (2) decides whether each batch row's query and key ids are
// non-decreasing (boundaries that pass their checks give non-decreasing ids by construction;
// given ids are checked, one block per row).  A tile pass then (3) for every 64-row
// query tile writes the key range [lo, hi) its rows can see, and for every 64-key tile the
// query range that can see it, intersected with the causal and window bounds, and (4) for
// every 128-row query tile and 128-key tile (the CTAs of the tensor-core kernels) writes its
// tile class and its visible pairs.  A second kernel sorts the tiles into longest-first work
// lists, which the tensor-core grids follow (MaxText commit message quoted on tokamax PR #1121:
// packed rows with segments of very different lengths, run starts per row).
// With non-decreasing ids a segment is one contiguous run: read straight from the boundaries
// with cu_seqlens, found by binary search in given ids; with arbitrary ids the ranges fall back
// to the causal/window bounds alone and the kernels test id equality pair by pair.  An empty range is stored as {n, 0} so that the union of
// two tile ranges (min of lo, max of hi) ignores it.
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

// Row pass.  With cu_seqlens (B == 1): a grid over the tokens, the boundaries in shared memory,
// block 0 checking them (a failed check is recorded in the status word and leaves the ids
// marked unsorted, so that the kernels compare ids pair by pair and every access stays inside
// its array).  With given ids: one block per batch row checks their order.
constexpr int kRowsTokensPerBlock = 4096;
__global__ void __launch_bounds__(1024) meta_rows_kernel(Params p, const int *cu, const int *cu_k, int nseq,
                                                         int *seg_out, int *segk_out, int *qoff_out,
                                                         int *koff_out, unsigned char *mono) {
  const int b = blockIdx.y;
  if (cu) {
    // The boundaries in shared memory when they fit: every token below searches them.
    constexpr int kCuSmem = 4096;
    __shared__ int cu_s[kCuSmem], cuk_s[kCuSmem];
    if (nseq + 1 <= kCuSmem) {
      for (int x = threadIdx.x; x <= nseq; x += blockDim.x) {
        cu_s[x] = cu[x];
        if (cu_k) cuk_s[x] = cu_k[x];
      }
      __syncthreads();
      cu = cu_s;
      if (cu_k) cu_k = cuk_s;
    }
    if (blockIdx.x == 0) {
      const int bad = __syncthreads_or(bad_bounds(cu, nseq, p.Sq) || (cu_k && bad_bounds(cu_k, nseq, p.Sk)));
      if (threadIdx.x == 0) {
        if (bad) set_status(p.status, kStatusBadCuSeqlens);
        mono[0] = (unsigned char)!bad;
      }
    }
    const int t0 = blockIdx.x * kRowsTokensPerBlock;
    if (cu_k) {
      // Separate query and key boundaries: ids per axis, and per token the bottom-right
      // offset end_k(s) - end_q(s) of its sequence.
      for (int t = t0 + threadIdx.x; t < min(t0 + kRowsTokensPerBlock, p.Sq); t += blockDim.x) {
        const int sq = seq_of(cu, nseq, t);
        seg_out[t] = sq;
        qoff_out[t] = seq_end(cu_k, nseq, p.Sk, sq) - seq_end(cu, nseq, p.Sq, sq);
      }
      for (int t = t0 + threadIdx.x; t < min(t0 + kRowsTokensPerBlock, p.Sk); t += blockDim.x) {
        const int sk = seq_of(cu_k, nseq, t);
        segk_out[t] = sk;
        koff_out[t] = seq_end(cu_k, nseq, p.Sk, sk) - seq_end(cu, nseq, p.Sq, sk);
      }
    } else {
      // Sq == Sk: one id array serves queries and keys.
      for (int t = t0 + threadIdx.x; t < min(t0 + kRowsTokensPerBlock, p.Sq); t += blockDim.x)
        seg_out[t] = seq_of(cu, nseq, t);
    }
    return;
  }
  const int *sq = p.seg_q + (size_t)b * p.Sq, *sk = p.seg_k + (size_t)b * p.Sk;
  int ok = 1;
  for (int i = threadIdx.x; i + 1 < p.Sq; i += blockDim.x) ok &= sq[i] <= sq[i + 1];
  for (int j = threadIdx.x; j + 1 < p.Sk; j += blockDim.x) ok &= sk[j] <= sk[j + 1];
  const int sorted = __syncthreads_and(ok);
  if (threadIdx.x == 0) mono[b] = (unsigned char)sorted;
}

// Per tile, after the row pass.  Grid: x over the tiles of one axis, y the batch row, z the
// axis (0: query tiles, 1: key tiles); 256 threads, each warp one 128-row tile.  With sorted ids
// every row's segment run on the other axis is read from the boundaries (cu_seqlens: sequence
// s spans [cu[s], cu[s + 1]) there, tokens at or past cu[nseq] forming sequence nseq) or found
// by binary search in given ids, in a shared-memory copy of the other axis's ids when they fit
// (a search in global memory pays a dependent load per step).
constexpr int kMetaSmemIds = 49152;  // ids copied to shared memory (192 KiB) at most
__global__ void __launch_bounds__(256) meta_tiles_kernel(Params p, const int *cu, const int *cu_k, int nseq,
                                                         const int *seg_out, const int *segk_out,
                                                         const int *qoff_out, const int *koff_out,
                                                         const unsigned char *mono, int2 *qrange, int2 *krange,
                                                         int4 *qtile, int4 *ktile, long long *qwork,
                                                         long long *kwork) {
  extern __shared__ int ids_s[];
  const int b = blockIdx.y;
  const bool qside = blockIdx.z == 0;
  const int *sq, *sk;
  if (cu) {
    sq = seg_out;
    sk = cu_k ? segk_out : seg_out;
  } else {
    sq = p.seg_q + (size_t)b * p.Sq;
    sk = p.seg_k + (size_t)b * p.Sk;
  }
  const bool sorted = mono[b] != 0;
  const int n_rows = qside ? p.Sq : p.Sk, n_other = qside ? p.Sk : p.Sq;
  const int *own = qside ? sq : sk;       // this axis's ids
  const int *other = qside ? sk : sq;     // the axis searched
  // boundaries of the other axis (cu_seqlens)
  const int *cu_other = cu ? (qside ? (cu_k ? cu_k : cu) : cu) : nullptr;
  if (sorted && !cu && n_other <= kMetaSmemIds) {
    for (int x = threadIdx.x; x < n_other; x += blockDim.x) ids_s[x] = other[x];
    __syncthreads();
    other = ids_s;
  }

  const bool per_seq = cu && cu_k;
  const int off = p.Sk - p.Sq;
  const int n64 = (n_rows + 63) / 64;

  // Tile classes and work of the 128-row query tiles (forward CTAs) and 128-key tiles
  // (backward CTAs), one warp per tile: every row's visible interval (causal / window bounds
  // at its offset, its segment's run when the ids are sorted), their union and intersection,
  // and the sum of their lengths -- the tile's visible pairs per head (an upper bound with
  // unsorted ids, where the kernels test pairs one by one and no tile is FULL).  The unions of
  // the two 64-row halves are the 64-granular ranges the FFMA kernels use.
  const int lane = threadIdx.x & 31;
  const int n128 = (n_rows + 127) / 128;
  const int tt = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tt < n128) {
    int lo_min = INT_MAX, hi_max = INT_MIN, lo_max = INT_MIN, hi_min = INT_MAX;
    int h_lo[2] = {INT_MAX, INT_MAX}, h_hi[2] = {INT_MIN, INT_MIN};  // per 64-row half
    long long work = 0;
    for (int r = tt * 128 + lane; r < min(tt * 128 + 128, n_rows); r += 32) {
      int lo, hi;
      if (qside) {
        const int ip = r + (per_seq ? qoff_out[r] : off);  // position on the key axis
        lo = p.window > 0 ? ip - p.window + 1 : 0;
        hi = p.causal ? ip + 1 : p.Sk;
      } else {
        const int kp = r - (per_seq ? koff_out[r] : off);  // position on the query axis
        lo = p.causal ? kp : 0;
        hi = p.window > 0 ? kp + p.window : p.Sq;
      }
      if (sorted) {
        const int id = own[r];
        if (cu_other) {  // checked boundaries: id in [0, nseq], cu_other non-decreasing, within n_other
          lo = max(lo, __ldg(cu_other + id));
          hi = min(hi, id < nseq ? __ldg(cu_other + id + 1) : n_other);
        } else {
          lo = max(lo, lower_bound_i(other, n_other, id));
          hi = min(hi, upper_bound_i(other, n_other, id));
        }
      }
      lo = max(lo, 0);
      hi = min(hi, n_other);
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
        (qside ? qrange : krange)[(size_t)b * n64 + t64] =
            h_lo[hf] < h_hi[hf] ? make_int2(h_lo[hf], h_hi[hf]) : make_int2(n_other, 0);
    }
    lo_min = __reduce_min_sync(0xffffffffu, lo_min);
    hi_max = __reduce_max_sync(0xffffffffu, hi_max);
    lo_max = __reduce_max_sync(0xffffffffu, lo_max);
    hi_min = __reduce_min_sync(0xffffffffu, hi_min);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) work += __shfl_xor_sync(0xffffffffu, work, o);
    if (lane == 0) {
      // A key tile that runs past Sk has no FULL query steps: the backward kernel computes P
      // for its missing keys too, and only the mask keeps them out (as the kernel's own
      // per-key intersection would, those keys seeing nothing).  Query rows past Sq are never
      // stored, so a query tile's class ignores them.
      const bool full_ok = sorted && (qside || tt * 128 + 128 <= p.Sk);
      const int4 c = lo_min < hi_max ? make_int4(lo_min, hi_max, full_ok ? lo_max : 0, full_ok ? hi_min : 0)
                                     : make_int4(n_other, 0, 0, 0);
      (qside ? qtile : ktile)[(size_t)b * n128 + tt] = c;
      (qside ? qwork : kwork)[(size_t)b * n128 + tt] = work;
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
  const int row_blocks = cu_seqlens ? (std::max(p.Sq, p.Sk) + kRowsTokensPerBlock - 1) / kRowsTokensPerBlock : 1;
  if (p.B > 65535) return cudaErrorInvalidValue;
  meta_rows_kernel<<<dim3((unsigned)std::max(row_blocks, 1), (unsigned)p.B), 1024, 0, st>>>(
      p, cu_seqlens, cu_seqlens_k, nseq, o.seg_q, o.seg_k, o.qoff, o.koff, o.mono);
  cudaError_t e = counted(cudaGetLastError());
  if (e != cudaSuccess) return e;
  {
    // blocks along x: enough warps for the 128-granular tiles of the longer axis (eight per
    // block), which also covers its 64-granular ranges (256 per block)
    const long long blocks = ((long long)(std::max(p.Sq, p.Sk) + 127) / 128 + 7) / 8;
    if (blocks > 0x7fffffffLL || p.B > 65535) return cudaErrorInvalidValue;
    const int n_ids = std::max(p.Sq, p.Sk);
    const size_t smem = (!cu_seqlens && n_ids <= kMetaSmemIds) ? (size_t)n_ids * sizeof(int) : 0;
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(meta_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    meta_tiles_kernel<<<dim3((unsigned)blocks, (unsigned)p.B, 2), 256, smem, st>>>(
        p, cu_seqlens, cu_seqlens_k, nseq, o.seg_q, o.seg_k, o.qoff, o.koff, o.mono, o.qrange, o.krange, o.qtile, o.ktile,
        o.qwork, o.kwork);
    e = counted(cudaGetLastError());
  }
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
