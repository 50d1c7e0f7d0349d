// splitkv.cu -- merge of a split-KV forward: each split s of a query row produced its own
// normalised output O_s and log-normaliser LSE_s over its share of the keys, without the sink
// column.  The row's statistics are those of the union of the splits plus that column, added
// exactly once here (TransformerEngine PR #3551, "What changed", second item, and the author's
// correction: merging tiles whose statistics each include the sink counts it once per tile):
//   LSE = ln( sum_s exp(LSE_s) + [sink or off-by-one column ? exp(its logit) : 0] )
//   O   = sum_s exp(LSE_s - LSE) O_s
// A row with no visible key in any split and no extra column keeps LSE = -inf and O = 0.
// Memory-bound: one warp per query row reads kv_splits partial rows (fp32) and writes one.
#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kMergeWarps = 8;

template <typename T>
__device__ __forceinline__ void store4(T *dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 o;
  o.x = *reinterpret_cast<uint32_t *>(&lo);
  o.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(dst) = o;
}

// grid: ceil(B * Hq * Sq / kMergeWarps) blocks of kMergeWarps warps; warp w -> row (b, h, i)
// in LSE order.  Lanes hold four consecutive d values per 128-wide slice of the row.
__global__ void __launch_bounds__(kMergeWarps * 32) splitkv_merge_kernel(Params p) {
  const int lane = threadIdx.x & 31;
  const size_t nrows = (size_t)p.B * p.Hq * p.Sq;
  const size_t row = (size_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (row >= nrows) return;
  const int i = (int)(row % p.Sq);
  const int h = (int)((row / p.Sq) % p.Hq);
  const int b = (int)(row / ((size_t)p.Sq * p.Hq));
  const int ns = p.kv_splits;
  // Largest log-normaliser among the splits and the extra column (natural log).
  const bool col = has_sink_col(p);
  float m = col ? sink_logit(p, h) : -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, p.lse_part[(size_t)s * nrows + row]);
  float z = 0.f;
  if (m != -INFINITY) {
    z = col ? expf(sink_logit(p, h) - m) : 0.f;
    for (int s = 0; s < ns; ++s) z += expf(p.lse_part[(size_t)s * nrows + row] - m);
  }
  const float lse = (m == -INFINITY) ? -INFINITY : m + logf(z);
  const int D = p.D;
  __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.O) + (((size_t)b * p.Sq + i) * p.Hq + h) * D;
  for (int d0 = 4 * lane; d0 < D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != -INFINITY) {
      for (int s = 0; s < ns; ++s) {
        const float ls = p.lse_part[(size_t)s * nrows + row];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - lse);
        const float4 x = *reinterpret_cast<const float4 *>(p.o_part + ((size_t)s * nrows + row) * D + d0);
        acc.x = fmaf(w, x.x, acc.x);
        acc.y = fmaf(w, x.y, acc.y);
        acc.z = fmaf(w, x.z, acc.z);
        acc.w = fmaf(w, x.w, acc.w);
      }
    }
    store4<__nv_bfloat16>(orow + d0, acc.x, acc.y, acc.z, acc.w);
  }
  if (lane == 0) p.LSE[row] = lse;
}

}  // namespace

cudaError_t launch_splitkv_merge(const Params &p, cudaStream_t st) {
  const size_t nrows = (size_t)p.B * p.Hq * p.Sq;
  const size_t blocks = (nrows + kMergeWarps - 1) / kMergeWarps;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffu) return cudaErrorInvalidValue;
  splitkv_merge_kernel<<<(unsigned)blocks, kMergeWarps * 32, 0, st>>>(p);
  return counted(cudaGetLastError());
}

}  // namespace attn
