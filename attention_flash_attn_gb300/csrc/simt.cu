// simt.cu -- fp32 CUDA-core (FFMA) attention kernels: forward, dQ and dK/dV.
//
// These carry every feature of the library (bias, soft-cap, sink, GQA, causal, window,
// segments) with accurate expf / expm1f / logf, for fp32 inputs (where a tensor-core
// tf32 product could not meet a 1e-5 relative error) and for calls with an additive bias.
// One warp owns one query row (forward, dQ) or one key row (dK/dV); K/V (or Q/dO) tiles
// are staged through shared memory as fp32.  The online softmax starts from the sink or the
// off-by-one column (m = its logit, l = 1) so that column enters each row exactly once.
#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kWarps = 8;     // rows per block
constexpr int kTile = 32;     // keys (or queries) per shared-memory tile
constexpr int kMaxPerLane = 16;  // D <= 512 -> at most 16 dims per lane (head dims above 256
                                 // exist only here: the dot products loop over D in shared
                                 // memory, the lane-owned accumulators cover D in 32-wide slices)

// Dims owned by this lane: lane, lane + 32, ... below D (unrolled so the arrays stay in
// registers).
#define FOR_LANE_DIMS(t2) \
  _Pragma("unroll") for (int t2 = 0; t2 < kMaxPerLane; ++t2) if (lane + 32 * t2 < D)

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__device__ __forceinline__ const T *q_ptr(const Params &p, int b, int i, int h) {
  return static_cast<const T *>(p.q) + b * p.q_sb + i * p.q_ss + h * p.q_sh;
}
template <typename T>
__device__ __forceinline__ const T *k_ptr(const Params &p, int b, int j, int g) {
  return static_cast<const T *>(p.k) + b * p.k_sb + j * p.k_ss + g * p.k_sh;
}
template <typename T>
__device__ __forceinline__ const T *v_ptr(const Params &p, int b, int j, int g) {
  return static_cast<const T *>(p.v) + b * p.v_sb + j * p.v_ss + g * p.v_sh;
}
__device__ __forceinline__ size_t row_off(const Params &p, int b, int i, int h) {
  return (((size_t)b * p.Sq + i) * p.Hq + h) * p.D;
}

// Pre-cap logit -> capped logit t and the backward factor.
template <typename T>
__device__ __forceinline__ void score(const Params &p, float s, int b, int h, int i, int j,
                                      float &t, float &factor) {
  float u = s * p.scale;
  if (p.bias) {
    const T *bp = static_cast<const T *>(p.bias);
    u += to_f(bp[b * p.bias_sb + h * p.bias_sh + (long long)i * p.Sk + j]);
  }
  if (p.cap > 0.f) {
    softcap_accurate(u, p.cap, p.inv_cap, t, factor);
  } else {
    t = u;
    factor = 1.f;
  }
}

// Key range [lo, hi) that rows [i0, i1] of batch b can see (a superset; per-pair
// visibility is still checked).
__device__ __forceinline__ void key_range(const Params &p, int b, int i0, int i1, int &lo, int &hi) {
  lo = 0;
  hi = p.Sk;
  if (!p.qoff) {  // per-sequence offsets: the tile ranges below carry the causal / window bounds
    if (p.causal) hi = min(hi, qpos(p, i1) + 1);
    if (p.window > 0) lo = max(lo, qpos(p, i0) - p.window + 1);
  }
  if (p.qrange) {
    const int nt = (p.Sq + 63) / 64;
    int2 a = p.qrange[(size_t)b * nt + i0 / 64], c = p.qrange[(size_t)b * nt + i1 / 64];
    lo = max(lo, min(a.x, c.x));
    hi = min(hi, max(a.y, c.y));
  }
}

// Query range [lo, hi) that can see keys [j0, j1] of batch b (a superset).
__device__ __forceinline__ void query_range(const Params &p, int b, int j0, int j1, int &lo, int &hi) {
  lo = 0;
  hi = p.Sq;
  if (!p.koff) {
    const int off = p.Sk - p.Sq;
    if (p.causal) lo = max(lo, j0 - off);
    if (p.window > 0) hi = min(hi, j1 - off + p.window);
  }
  if (p.krange) {
    const int nt = (p.Sk + 63) / 64;
    int2 a = p.krange[(size_t)b * nt + j0 / 64], c = p.krange[(size_t)b * nt + j1 / 64];
    lo = max(lo, min(a.x, c.x));
    hi = min(hi, max(a.y, c.y));
  }
}

// ---------------------------------------------------------------------------- forward
// grid (ceil(Sq/8), Hq, B), block 256.  smem: K [32][D+1], V [32][D], Q [8][D] fp32.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(Params p) {
  extern __shared__ float sm[];
  const int D = p.D, Dp = D + 1;
  float *Ks = sm;
  float *Vs = Ks + kTile * Dp;
  float *Qs = Vs + kTile * D;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, h = blockIdx.y, g = h / p.G;
  const int i0 = blockIdx.x * kWarps;
  const int i1 = min(i0 + kWarps, p.Sq) - 1;
  const int i = i0 + warp;
  const bool row_ok = i < p.Sq;
  for (int d = lane; d < D; d += 32)
    Qs[warp * D + d] = row_ok ? to_f(q_ptr<T>(p, b, i, h)[d]) : 0.f;

  int lo, hi;
  key_range(p, b, i0, i1, lo, hi);
  float m = has_sink_col(p) ? sink_logit(p, h) : -INFINITY;
  float l = has_sink_col(p) ? 1.f : 0.f;
  float acc[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) acc[t] = 0.f;

  for (int j0 = lo; j0 < hi; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
      const int jj = e / D, d = e % D, j = j0 + jj;
      const bool ok = j < p.Sk;
      Ks[jj * Dp + d] = ok ? to_f(k_ptr<T>(p, b, j, g)[d]) : 0.f;
      Vs[jj * D + d] = ok ? to_f(v_ptr<T>(p, b, j, g)[d]) : 0.f;
    }
    __syncthreads();
    const int j = j0 + lane;
    float t = -INFINITY;
    const bool vis = row_ok && j < hi && visible(p, b, i, j);
    if (vis) {
      float s = 0.f;
      for (int d = 0; d < D; ++d) s = fmaf(Qs[warp * D + d], Ks[lane * Dp + d], s);
      float f;
      score<T>(p, s, b, h, i, j, t, f);
    }
    const float mn = fmaxf(m, warp_max(t));
    const float alpha = (mn == -INFINITY) ? 0.f : expf(m - mn);
    const float pj = vis ? expf(t - mn) : 0.f;
    l = l * alpha + warp_sum(pj);
    FOR_LANE_DIMS(t2) acc[t2] *= alpha;
    for (int jj = 0; jj < kTile; ++jj) {
      const float pjj = __shfl_sync(0xffffffffu, pj, jj);
      if (pjj != 0.f)
        FOR_LANE_DIMS(t2) acc[t2] = fmaf(pjj, Vs[jj * D + lane + 32 * t2], acc[t2]);
    }
    m = mn;
  }
  if (!row_ok) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T *O = static_cast<T *>(p.O) + row_off(p, b, i, h);
  FOR_LANE_DIMS(t2) O[lane + 32 * t2] = from_f<T>(acc[t2] * inv);
  if (lane == 0) p.LSE[((size_t)b * p.Hq + h) * p.Sq + i] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ---------------------------------------------------------------------------- dQ (+ dbias)
// grid (ceil(Sq/8), Hq, B), block 256.  smem: K [32][D+1], V [32][D+1], Q [8][D], dO [8][D].
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dq_kernel(Params p) {
  extern __shared__ float sm[];
  const int D = p.D, Dp = D + 1;
  float *Ks = sm;
  float *Vs = Ks + kTile * Dp;
  float *Qs = Vs + kTile * Dp;
  float *dOs = Qs + kWarps * D;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, h = blockIdx.y, g = h / p.G;
  const int i0 = blockIdx.x * kWarps;
  const int i1 = min(i0 + kWarps, p.Sq) - 1;
  const int i = i0 + warp;
  const bool row_ok = i < p.Sq;
  const T *dO = static_cast<const T *>(p.dO);
  for (int d = lane; d < D; d += 32) {
    Qs[warp * D + d] = row_ok ? to_f(q_ptr<T>(p, b, i, h)[d]) : 0.f;
    dOs[warp * D + d] = row_ok ? to_f(dO[row_off(p, b, i, h) + d]) : 0.f;
  }
  const size_t ri = ((size_t)b * p.Hq + h) * p.Sq + (row_ok ? i : 0);
  const float lse = row_ok ? p.LSE[ri] : -INFINITY;
  const float Di = row_ok ? p.Dvec[((size_t)b * p.Hq + h) * p.sq_pad + i] : 0.f;
  const bool live = row_ok && lse != -INFINITY;

  int lo, hi;
  key_range(p, b, i0, i1, lo, hi);
  float acc[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) acc[t] = 0.f;

  for (int j0 = lo; j0 < hi; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
      const int jj = e / D, d = e % D, j = j0 + jj;
      const bool ok = j < p.Sk;
      Ks[jj * Dp + d] = ok ? to_f(k_ptr<T>(p, b, j, g)[d]) : 0.f;
      Vs[jj * Dp + d] = ok ? to_f(v_ptr<T>(p, b, j, g)[d]) : 0.f;
    }
    __syncthreads();
    const int j = j0 + lane;
    float ds = 0.f;
    if (live && j < hi && visible(p, b, i, j)) {
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < D; ++d) {
        s = fmaf(Qs[warp * D + d], Ks[lane * Dp + d], s);
        dp = fmaf(dOs[warp * D + d], Vs[lane * Dp + d], dp);
      }
      float t, f;
      score<T>(p, s, b, h, i, j, t, f);
      const float pij = expf(t - lse);
      ds = pij * (dp - Di) * f;
      if (p.dbias_acc) {
        const int bb = p.bias_B == 1 ? 0 : b, hb = p.bias_H == 1 ? 0 : h;
        atomicAdd(p.dbias_acc + (((size_t)bb * p.bias_H + hb) * p.Sq + i) * p.Sk + j, ds);
      }
    }
    for (int jj = 0; jj < kTile; ++jj) {
      const float d2 = __shfl_sync(0xffffffffu, ds, jj);
      if (d2 != 0.f)
        FOR_LANE_DIMS(t2) acc[t2] = fmaf(d2, Ks[jj * Dp + lane + 32 * t2], acc[t2]);
    }
  }
  if (!row_ok) return;
  T *dQ = static_cast<T *>(p.dQ) + row_off(p, b, i, h);
  FOR_LANE_DIMS(t2) dQ[lane + 32 * t2] = from_f<T>(acc[t2] * p.scale);
}

// ---------------------------------------------------------------------------- dK, dV
// One warp per key j of kv head g; loops over the G query heads of the group and the
// query rows that can see the block's keys.
// grid (ceil(Sk/8), Hkv, B), block 256.  smem: Q [32][D+1], dO [32][D+1], K [8][D], V [8][D],
// lse/D [32] x 2.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dkdv_kernel(Params p) {
  extern __shared__ float sm[];
  const int D = p.D, Dp = D + 1;
  float *Qs = sm;
  float *dOs = Qs + kTile * Dp;
  float *Kw = dOs + kTile * Dp;
  float *Vw = Kw + kWarps * D;
  float *Ls = Vw + kWarps * D;
  float *Ds = Ls + kTile;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, g = blockIdx.y;
  const int j0 = blockIdx.x * kWarps;
  const int j1 = min(j0 + kWarps, p.Sk) - 1;
  const int j = j0 + warp;
  const bool col_ok = j < p.Sk;
  for (int d = lane; d < D; d += 32) {
    Kw[warp * D + d] = col_ok ? to_f(k_ptr<T>(p, b, j, g)[d]) : 0.f;
    Vw[warp * D + d] = col_ok ? to_f(v_ptr<T>(p, b, j, g)[d]) : 0.f;
  }
  int lo, hi;
  query_range(p, b, j0, j1, lo, hi);
  float dk[kMaxPerLane], dv[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) dk[t] = dv[t] = 0.f;
  const T *dO = static_cast<const T *>(p.dO);

  for (int h = g * p.G; h < (g + 1) * p.G; ++h) {
    for (int r0 = lo; r0 < hi; r0 += kTile) {
      __syncthreads();
      for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int ii = e / D, d = e % D, i = r0 + ii;
        const bool ok = i < hi;
        Qs[ii * Dp + d] = ok ? to_f(q_ptr<T>(p, b, i, h)[d]) : 0.f;
        dOs[ii * Dp + d] = ok ? to_f(dO[row_off(p, b, i, h) + d]) : 0.f;
      }
      if (threadIdx.x < kTile) {
        const int i = r0 + threadIdx.x;
        const bool ok = i < hi;
        Ls[threadIdx.x] = ok ? p.LSE[((size_t)b * p.Hq + h) * p.Sq + i] : -INFINITY;
        Ds[threadIdx.x] = ok ? p.Dvec[((size_t)b * p.Hq + h) * p.sq_pad + i] : 0.f;
      }
      __syncthreads();
      const int i = r0 + lane;
      float pij = 0.f, ds = 0.f;
      if (col_ok && i < hi && Ls[lane] != -INFINITY && visible(p, b, i, j)) {
        float s = 0.f, dp = 0.f;
        for (int d = 0; d < D; ++d) {
          s = fmaf(Qs[lane * Dp + d], Kw[warp * D + d], s);
          dp = fmaf(dOs[lane * Dp + d], Vw[warp * D + d], dp);
        }
        float t, f;
        score<T>(p, s, b, h, i, j, t, f);
        pij = expf(t - Ls[lane]);
        ds = pij * (dp - Ds[lane]) * f;
      }
      for (int ii = 0; ii < kTile; ++ii) {
        const float pp = __shfl_sync(0xffffffffu, pij, ii);
        const float d2 = __shfl_sync(0xffffffffu, ds, ii);
        if (pp != 0.f)
          FOR_LANE_DIMS(t2) {
            dv[t2] = fmaf(pp, dOs[ii * Dp + lane + 32 * t2], dv[t2]);
            dk[t2] = fmaf(d2, Qs[ii * Dp + lane + 32 * t2], dk[t2]);
          }
      }
    }
  }
  if (!col_ok) return;
  const size_t off = (((size_t)b * p.Sk + j) * p.Hkv + g) * p.D;
  T *dK = static_cast<T *>(p.dK) + off;
  T *dV = static_cast<T *>(p.dV) + off;
  FOR_LANE_DIMS(t2) {
    dK[lane + 32 * t2] = from_f<T>(dk[t2] * p.scale);
    dV[lane + 32 * t2] = from_f<T>(dv[t2]);
  }
}

template <typename T>
cudaError_t launch_all_fwd(const Params &p, cudaStream_t st) {
  const int D = p.D;
  size_t sm = sizeof(float) * (kTile * (D + 1) + kTile * D + kWarps * D);  // 148 KiB at D = 512
  // Set on every call: cheap, idempotent, and per device.
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Sq + kWarps - 1) / kWarps, p.Hq, p.B);
  simt_fwd_kernel<T><<<grid, kWarps * 32, sm, st>>>(p);
  return counted(cudaGetLastError());
}

template <typename T>
cudaError_t launch_all_bwd(const Params &p, cudaStream_t st) {
  const int D = p.D;
  const size_t sm_dq = sizeof(float) * (2 * kTile * (D + 1) + 2 * kWarps * D);              // 160 KiB at D = 512
  const size_t sm_kv = sizeof(float) * (2 * kTile * (D + 1) + 2 * kWarps * D + 2 * kTile);  // 161 KiB
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_dq_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_dq);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(simt_bwd_dkdv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_kv);
  if (e != cudaSuccess) return e;
  dim3 g1((p.Sq + kWarps - 1) / kWarps, p.Hq, p.B);
  simt_bwd_dq_kernel<T><<<g1, kWarps * 32, sm_dq, st>>>(p);
  e = counted(cudaGetLastError());
  if (e != cudaSuccess) return e;
  if (p.Sk == 0) return cudaSuccess;  // no keys: no dK / dV
  dim3 g2((p.Sk + kWarps - 1) / kWarps, p.Hkv, p.B);
  simt_bwd_dkdv_kernel<T><<<g2, kWarps * 32, sm_kv, st>>>(p);
  return counted(cudaGetLastError());
}

}  // namespace

cudaError_t simt_forward(const Params &p, int dtype, cudaStream_t st) {
  return dtype == kF32 ? launch_all_fwd<float>(p, st) : launch_all_fwd<__nv_bfloat16>(p, st);
}

cudaError_t simt_backward(const Params &p, int dtype, cudaStream_t st) {
  return dtype == kF32 ? launch_all_bwd<float>(p, st) : launch_all_bwd<__nv_bfloat16>(p, st);
}

}  // namespace attn
