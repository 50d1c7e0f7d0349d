// bwd_score.cuh -- the backward's element-wise score function, shared by the tensor-core
// backward kernels: from a raw score the (capped, biased) logit in log2 units less the row's
// LSE, and the cap's chain-rule factor, as packed pairs; and the predicated fp32 reduce-add
// that accumulates dbias.  The backward forms P = exp2(t log2(e) - LSE log2(e)) from the
// forward's LSE, so every backward kernel must use this one function.
#pragma once

#include "tc_common.cuh"

namespace attn {
namespace bwd_score {

using namespace tc;

constexpr float kLog2e = 1.4426950408889634f;

// Score constants of the element-wise backward, as packed pairs.  With the soft-cap,
// e = exp(2 u / cap) for u = scale s, r = 1 / (1 + e), so tanh(u / cap) = 1 - 2 r and
// 1 - tanh^2 = 4 r (1 - r) = 4 e r^2; the capped logit in log2 units is cap log2(e) (1 - 2 r).
// The exponent is clamped at 126 (a huge e gives r ~ 0, tanh = 1, and e r^2 = 0 rather than
// inf * 0); an underflowing e gives r = 1 (tanh = -1).
// With a bias the logit is u = scale s + bias: the bias enters as its own term (bin: its
// factor, 2 log2(e) / cap with the cap, log2(e) without), and the chain-rule factor is formed
// without the softmax scale (f4 = 4, fone = 1), so that dU = P (dP - D) f -- the bias's own
// gradient -- is at hand before the scale is applied for dS.
struct BwdScore {
  uint64_t cin, one, mcap2, cap2, fs, sc2, scale, bin, f4;
  __device__ BwdScore(float scale_, float inv_cap, float cap) {
    cin = f2_splat(2.f * kLog2e * scale_ * inv_cap);
    one = f2_splat(1.f);
    mcap2 = f2_splat(-2.f * cap * kLog2e);
    cap2 = f2_splat(cap * kLog2e);
    fs = f2_splat(4.f * scale_);
    sc2 = f2_splat(scale_ * kLog2e);
    scale = f2_splat(scale_);
    bin = f2_splat(cap > 0.f ? 2.f * kLog2e * inv_cap : kLog2e);
    f4 = f2_splat(4.f);
  }
};

// The bias of one bf16 pair (low half first) as a pair of floats.
__device__ __forceinline__ uint64_t bias_pair(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// dbias accumulation: dU of this thread's key for the visible queries of a chunk, added into
// the fp32 accumulator (reduce-adds: broadcast dimensions and GQA heads may share elements).
// Predicated in the instruction itself, so that per-lane visibility never splits the warp
// ahead of the tensor-memory instructions, which need it converged.
__device__ __forceinline__ void red_add_f32_if(float *addr, float v, uint32_t pred) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p red.global.add.f32 [%0], %1;\n\t}" ::"l"(addr),
               "f"(v), "r"(pred)
               : "memory");
}

// One pair of raw scores -> (t2 - LSE2, f): t2 the (capped) logit in log2 units, f the
// cap's chain-rule factor times the softmax scale.  FRCP: the cap's reciprocal on the FMA pipe
// (f2_sigmoid2_neg); otherwise ex2 + rcp on the special-function unit.  The head-dim-256 dK pass
// keeps the latter: its element-wise work sits on the S^T -> dP^T dependency chain and is not
// bound by the special-function unit, and the longer FMA sequence measured 5 % slower there.
// BIAS: b2 is the pair's bias, and f comes without the softmax scale.
template <bool CAP, bool FRCP, bool BIAS = false>
__device__ __forceinline__ void score_pair(uint32_t s0, uint32_t s1, uint64_t lse2, const BwdScore &k, uint64_t &y,
                                           uint64_t &f, uint64_t b2 = 0) {
  const uint64_t s2 = f2_pack(__uint_as_float(s0), __uint_as_float(s1));
  if constexpr (CAP) {
    uint64_t r2, e2;
    const uint64_t x2 = BIAS ? f2_fma(s2, k.cin, f2_mul(b2, k.bin)) : f2_mul(s2, k.cin);
    if constexpr (FRCP) {
      r2 = f2_sigmoid2_neg(x2, e2);
    } else {
      float xa, xb, da, db;
      f2_unpack(x2, xa, xb);
      e2 = f2_pack(ex2_approx(fminf(xa, 126.f)), ex2_approx(fminf(xb, 126.f)));
      f2_unpack(f2_add(e2, k.one), da, db);
      r2 = f2_pack(rcp_approx(da), rcp_approx(db));
    }
    y = f2_sub(f2_fma(r2, k.mcap2, k.cap2), lse2);
    // 1 - tanh^2 = 4 r (1 - r) = 4 e r^2: the second form keeps full relative accuracy where the
    // cap saturates (r -> 1, where 1 - r would cancel), so the tiny gradients there stay right.
    f = f2_mul(f2_mul(e2, BIAS ? k.f4 : k.fs), f2_mul(r2, r2));
  } else {
    y = f2_sub(BIAS ? f2_fma(s2, k.sc2, f2_mul(b2, k.bin)) : f2_mul(s2, k.sc2), lse2);
    f = BIAS ? k.one : k.scale;
  }
}
__device__ __forceinline__ uint64_t ex2_pair(uint64_t y) {
  float a, b;
  f2_unpack(y, a, b);
  return f2_pack(ex2_approx(a), ex2_approx(b));
}
__device__ __forceinline__ uint32_t bf16_pair(uint64_t v) {
  float a, b;
  f2_unpack(v, a, b);
  return pack_bf16(a, b);
}

}  // namespace bwd_score
}  // namespace attn
