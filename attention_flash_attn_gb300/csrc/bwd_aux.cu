// bwd_aux.cu -- memory-bound pieces of the backward pass.
//
// bwd_pre:  D_i = sum_d dO_i[d] * O_i[d] (fp32) for every (b, h, i), and, for the
//           tensor-core backward, LSE_i * log2(e), both in rows padded to a multiple of 128
//           so that the backward can fetch them with bulk copies; the sink gradient's
//           per-block partial sums -sum_i exp(sink_h - LSE_i) * D_i; and, when the
//           tensor-core backward accumulates dQ in fp32, zeroing of that accumulator.
//           The sink gradient follows TransformerEngine PR #3551 ("What changed"): the
//           sink column's probability times (0 - D_i), summed over every row and batch.
// bwd_post: the fp32 dQ accumulator converted to the output dtype, the deterministic
//           final dsink reduction (fixed order), and the fp32 dbias accumulator written
//           out in the bias dtype.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

// Query positions per preprocess block: 64, halved down to 16 while the grid would not fill two
// blocks per SM (chunked-prefill and decode-like shapes: few rows, few heads).
constexpr int kPreRowsMax = 64, kPreRowsMin = 16;
constexpr int kPreWarps = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 16-byte vector dot of dO and O rows.
template <typename T>
__device__ __forceinline__ float chunk_dot(const T *a, const T *b);
template <>
__device__ __forceinline__ float chunk_dot<__nv_bfloat16>(const __nv_bfloat16 *a, const __nv_bfloat16 *b) {
  uint4 x = *reinterpret_cast<const uint4 *>(a), y = *reinterpret_cast<const uint4 *>(b);
  const __nv_bfloat162 *xa = reinterpret_cast<const __nv_bfloat162 *>(&x);
  const __nv_bfloat162 *ya = reinterpret_cast<const __nv_bfloat162 *>(&y);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 fx = __bfloat1622float2(xa[k]), fy = __bfloat1622float2(ya[k]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}
template <>
__device__ __forceinline__ float chunk_dot<float>(const float *a, const float *b) {
  float4 x = *reinterpret_cast<const float4 *>(a), y = *reinterpret_cast<const float4 *>(b);
  return fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w)));
}

// One query row's (dO, O) chunk pair: 16 bytes of each.
template <typename T>
__device__ __forceinline__ float chunk_dot_raw(const uint4 &x, const uint4 &y);
template <>
__device__ __forceinline__ float chunk_dot_raw<__nv_bfloat16>(const uint4 &x, const uint4 &y) {
  const __nv_bfloat162 *xa = reinterpret_cast<const __nv_bfloat162 *>(&x);
  const __nv_bfloat162 *ya = reinterpret_cast<const __nv_bfloat162 *>(&y);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fx = __bfloat1622float2(xa[k]), fy = __bfloat1622float2(ya[k]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}
template <>
__device__ __forceinline__ float chunk_dot_raw<float>(const uint4 &x, const uint4 &y) {
  return fmaf(__uint_as_float(x.x), __uint_as_float(y.x),
              fmaf(__uint_as_float(x.y), __uint_as_float(y.y),
                   fmaf(__uint_as_float(x.z), __uint_as_float(y.z), __uint_as_float(x.w) * __uint_as_float(y.w))));
}

// -D as three bf16 parts, in the first three of a row's eight bf16 slots (the other five
// zero): the row of the fused tensor-core backward's K = 16 operand that starts dP^T at -D.
// Each part is the bf16 rounding of what the ones before it left; every subtraction is exact
// in fp32 and the last remainder fits 8 bits, so the parts sum to -D exactly (barring
// underflow).
__device__ __forceinline__ uint4 neg_d_parts(float d) {
  const float x = -d;
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  return make_uint4((uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(mid) << 16),
                    (uint32_t)__bfloat16_as_ushort(lo), 0u, 0u);
}

// grid (ceil(Sq/ROWS), B, ceil(Hq/8)), block 256: warp w of z-block z handles head 8 z + w;
// rows in order, so the per-(block, head) partial sums are deterministic.  ROWS is a template
// parameter: the same kernel with a run-time row count measured 1.3 % slower on the D=64 sink
// workload's step.
//
// NC > 0 (a row is NC 16-byte chunks, NC dividing 32 or a multiple of it): a warp covers
// 32 / NC rows per load, one lane per chunk (NC > 32: one row, NC / 32 chunks per lane), and
// keeps kPreUnroll such loads in flight per lane before reducing each row over its lanes.
// NC == 0: any other row length, one row per warp at a time.
constexpr int kPreUnroll = 4;
template <typename T, int NC, int ROWS>
__global__ void __launch_bounds__(kPreWarps * 32) bwd_pre_kernel(Params p, int zero_dqacc) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.y;
  const int i0 = blockIdx.x * ROWS, i1 = min(i0 + ROWS, p.Sq);
  constexpr int per_chunk = 16 / sizeof(T);
  const T *O = static_cast<const T *>(p.O);
  const T *dO = static_cast<const T *>(p.dO);
  for (int h = blockIdx.z * kPreWarps + warp; h < p.Hq && h < (int)(blockIdx.z + 1) * kPreWarps; h += kPreWarps) {
    float part = 0.f;
    const float sink = p.sink ? p.sink[h] : 0.f;
    if constexpr (NC > 0) {
      // LPR lanes per row (NC > 32: the whole warp, CPL chunks per lane)
      constexpr int LPR = NC > 32 ? 32 : NC, CPL = NC > 32 ? NC / 32 : 1;
      constexpr int RPL = 32 / LPR;  // rows per warp-wide load
      const int sub = lane / LPR, c = lane % LPR;
      for (int ib = i0; ib < i1; ib += RPL * kPreUnroll) {
        uint4 xa[kPreUnroll][CPL], xb[kPreUnroll][CPL];
#pragma unroll
        for (int u = 0; u < kPreUnroll; ++u) {
          const int i = ib + u * RPL + sub;
#pragma unroll
          for (int cp = 0; cp < CPL; ++cp) {
            if (i < i1) {
              const size_t row = (((size_t)b * p.Sq + i) * p.Hq + h) * p.D + (size_t)(c + cp * LPR) * per_chunk;
              xa[u][cp] = __ldg(reinterpret_cast<const uint4 *>(dO + row));
              xb[u][cp] = __ldg(reinterpret_cast<const uint4 *>(O + row));
            } else {
              xa[u][cp] = xb[u][cp] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        float s[kPreUnroll];
#pragma unroll
        for (int u = 0; u < kPreUnroll; ++u) {
          s[u] = 0.f;
#pragma unroll
          for (int cp = 0; cp < CPL; ++cp) s[u] += chunk_dot_raw<T>(xa[u][cp], xb[u][cp]);
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) {
#pragma unroll
          for (int u = 0; u < kPreUnroll; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], o);
        }
#pragma unroll
        for (int u = 0; u < kPreUnroll; ++u) {
          const int i = ib + u * RPL + sub;
          if (i >= i1) continue;
          if (c == 0) {
            const size_t ri = ((size_t)b * p.Hq + h) * p.Sq + i;
            const size_t rp = ((size_t)b * p.Hq + h) * p.sq_pad + i;
            const float lse = p.LSE[ri];
            p.Dvec[rp] = s[u];
            if (p.lse2p) p.lse2p[rp] = lse * 1.4426950408889634f;
            if (p.dsplit) p.dsplit[rp] = neg_d_parts(s[u]);
            if (p.sink) part = fmaf(expf(sink - lse), s[u], part);
          }
          if (zero_dqacc) {
#pragma unroll
            for (int cp = 0; cp < CPL; ++cp) {
              float4 *z = reinterpret_cast<float4 *>(p.dQacc + (((size_t)b * p.Sq + i) * p.Hq + h) * p.D +
                                                     (size_t)(c + cp * LPR) * per_chunk);
#pragma unroll
              for (int v = 0; v < per_chunk / 4; ++v) z[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
      }
      // Only the first lane of each row segment holds a partial sum: add them in a fixed order.
      part = warp_sum(part);
    } else {
      const int nchunk = p.D / per_chunk;
      for (int i = i0; i < i1; ++i) {
        const size_t row = (((size_t)b * p.Sq + i) * p.Hq + h) * p.D;
        float s = 0.f;
        for (int c = lane; c < nchunk; c += 32) s += chunk_dot<T>(dO + row + c * per_chunk, O + row + c * per_chunk);
        s = warp_sum(s);
        const size_t ri = ((size_t)b * p.Hq + h) * p.Sq + i;
        const size_t rp = ((size_t)b * p.Hq + h) * p.sq_pad + i;
        if (lane == 0) {
          p.Dvec[rp] = s;
          if (p.lse2p) p.lse2p[rp] = p.LSE[ri] * 1.4426950408889634f;
          if (p.dsplit) p.dsplit[rp] = neg_d_parts(s);
        }
        if (p.sink) part = fmaf(expf(sink - p.LSE[ri]), s, part);
        if (zero_dqacc) {
          float4 *z = reinterpret_cast<float4 *>(p.dQacc + row);
          for (int c = lane; c < p.D / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    if (p.sink && lane == 0)
      p.dsink_part[(size_t)h * p.n_part + (size_t)b * gridDim.x + blockIdx.x] = -part;
    // The last block of the row also fills the padding: D = 0, LSE = +inf (P = 0 there).
    if (i1 == p.Sq)
      for (int i = p.Sq + lane; i < p.sq_pad; i += 32) {
        const size_t rp = ((size_t)b * p.Hq + h) * p.sq_pad + i;
        p.Dvec[rp] = 0.f;
        if (p.lse2p) p.lse2p[rp] = INFINITY;
        if (p.dsplit) p.dsplit[rp] = make_uint4(0u, 0u, 0u, 0u);
      }
  }
}

// Eight fp32 values -> eight output values in one 16-byte store (bf16) or two (fp32).
template <typename T>
__device__ __forceinline__ void store8(T *dst, const float4 &x, const float4 &y);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *dst, const float4 &x, const float4 &y) {
  uint4 o;
  __nv_bfloat162 t;
  t = __floats2bfloat162_rn(x.x, x.y); o.x = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(x.z, x.w); o.y = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(y.x, y.y); o.z = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(y.z, y.w); o.w = *reinterpret_cast<uint32_t *>(&t);
  *reinterpret_cast<uint4 *>(dst) = o;
}
template <>
__device__ __forceinline__ void store8<float>(float *dst, const float4 &x, const float4 &y) {
  reinterpret_cast<float4 *>(dst)[0] = x;
  reinterpret_cast<float4 *>(dst)[1] = y;
}

template <typename T>
__global__ void __launch_bounds__(256) bwd_post_kernel(Params p, int convert_dq, size_t dbias_elems) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t gwarp = (size_t)blockIdx.x * 8 + warp;
  if (p.dsink && gwarp < (size_t)p.Hq) {
    const float *part = p.dsink_part + gwarp * p.n_part;
    float s = 0.f;
    for (int c = lane; c < p.n_part; c += 32) s += part[c];
    s = warp_sum(s);
    if (lane == 0) p.dsink[gwarp] = s;
  }
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthr = (size_t)gridDim.x * blockDim.x;
  if (convert_dq) {
    // D is a multiple of 8 and dQ 16-byte aligned: whole groups of eight.
    const size_t n8 = (size_t)p.B * p.Sq * p.Hq * p.D / 8;
    const float4 *src = reinterpret_cast<const float4 *>(p.dQacc);
    T *dst = static_cast<T *>(p.dQ);
    for (size_t e = tid; e < n8; e += nthr) store8<T>(dst + 8 * e, __ldg(src + 2 * e), __ldg(src + 2 * e + 1));
  }
  if (dbias_elems) {
    T *dst = static_cast<T *>(p.dbias);
    for (size_t e = tid; e < dbias_elems; e += nthr) dst[e] = from_f<T>(p.dbias_acc[e]);
  }
}

template <typename T>
cudaError_t launch_pre_t(const Params &p, bool zero_dqacc, cudaStream_t st) {
  // z: groups of kPreWarps heads (one per warp), so that heads spread over the SMs too
  const int rows = bwd_pre_rows(p.B, p.Sq, p.Hq);
  dim3 grid((p.Sq + rows - 1) / rows, p.B, (p.Hq + kPreWarps - 1) / kPreWarps);
  const int nc = p.D * (int)sizeof(T) / 16;
  auto go = [&](auto rc) {
    constexpr int R = decltype(rc)::value;
    switch (nc) {
      case 4: bwd_pre_kernel<T, 4, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
      case 8: bwd_pre_kernel<T, 8, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
      case 16: bwd_pre_kernel<T, 16, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
      case 32: bwd_pre_kernel<T, 32, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
      case 64: bwd_pre_kernel<T, 64, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
      default: bwd_pre_kernel<T, 0, R><<<grid, kPreWarps * 32, 0, st>>>(p, zero_dqacc); break;
    }
  };
  if (rows == 64) go(std::integral_constant<int, 64>());
  else if (rows == 32) go(std::integral_constant<int, 32>());
  else go(std::integral_constant<int, 16>());
  return counted(cudaGetLastError());
}

}  // namespace

int bwd_pre_rows(int B, int Sq, int Hq) {
  const long long z = (Hq + kPreWarps - 1) / kPreWarps, target = 2LL * device_sm_count();
  int rows = kPreRowsMax;
  while (rows > kPreRowsMin && (long long)((Sq + rows - 1) / rows) * B * z < target) rows /= 2;
  return rows;
}
int bwd_pre_partials(int B, int Sq, int Hq) {
  const int rows = bwd_pre_rows(B, Sq, Hq);
  return B * ((Sq + rows - 1) / rows);
}
int bwd_pre_partials_max(int B, int Sq) { return B * ((Sq + kPreRowsMin - 1) / kPreRowsMin); }

cudaError_t launch_bwd_pre(const Params &p, int dtype, bool zero_dqacc, cudaStream_t st) {
  return dtype == kF32 ? launch_pre_t<float>(p, zero_dqacc, st) : launch_pre_t<__nv_bfloat16>(p, zero_dqacc, st);
}

cudaError_t launch_bwd_post(const Params &p, int dtype, bool convert_dq, size_t dbias_elems,
                            cudaStream_t st) {
  size_t work = 0;
  if (convert_dq) work = (size_t)p.B * p.Sq * p.Hq * p.D / 8;
  if (dbias_elems > work) work = dbias_elems;
  size_t blocks = (work + 255) / 256;
  const size_t sink_blocks = p.dsink ? (size_t)(p.Hq + 7) / 8 : 0;
  if (blocks < sink_blocks) blocks = sink_blocks;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) return cudaSuccess;
  if (dtype == kF32)
    bwd_post_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(p, convert_dq, dbias_elems);
  else
    bwd_post_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(p, convert_dq, dbias_elems);
  return counted(cudaGetLastError());
}

}  // namespace attn
