// tc_common.cuh -- sm_100-family building blocks written as inline PTX: mbarriers with
// bounded waits, TMA tile loads, tensor-memory (TMEM) allocation, tcgen05 MMAs with their
// shared-memory and instruction descriptors, and TMEM <-> register moves.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is resolved at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {
namespace tc {

// ------------------------------------------------------------------ generic helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The first wait to give up also leaves where it was: words 1..6 of the status area hold a
// marker, the barrier's shared-memory offset and parity, and the CTA and thread indices.
__device__ __forceinline__ void record_timeout(unsigned *status, uint32_t bar, uint32_t parity) {
  if (!status) return;
  if (atomicCAS(status + 1, 0u, 1u) == 0u) {
    status[2] = bar;
    status[3] = parity;
    status[4] = blockIdx.x | (blockIdx.y << 16);
    status[5] = blockIdx.z;
    status[6] = threadIdx.x;
    __threadfence();
  }
  atomicOr(status, kStatusWaitTimeout);
}

__device__ __forceinline__ unsigned status_peek(const unsigned *status) {
  unsigned v = 0;
  if (status) asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(status));
  return v;
}

// Waits for the phase of parity `parity` to complete, for at most kWaitLimitNs.  Gives up
// early if another CTA has already recorded a timeout (so one fault cannot turn into every
// CTA timing out in turn).  Returns false, with kStatusWaitTimeout recorded, if it gave up.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
// Waits that give up inside the CTA that recorded the first timeout also leave, per warp,
// the barrier and parity they were waiting on (words 8 + 2 w, 9 + 2 w; w < 16).
__device__ __forceinline__ void record_abort(unsigned *status, uint32_t bar, uint32_t parity) {
  if (!status) return;
  const unsigned w = threadIdx.x >> 5;
  if (w < 16 && status[1] == 1u && status[4] == (blockIdx.x | (blockIdx.y << 16)) && status[5] == blockIdx.z) {
    status[8 + 2 * w] = bar;
    status[9 + 2 * w] = parity | 0x100u;
  }
}

// limit_ns: the kernels pass kWaitLimitNs; the self-test of this path passes a short limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (status_peek(status) & kStatusWaitTimeout) {
        record_abort(status, bar, parity);
        return false;
      }
      if (globaltimer_ns() - t0 > limit_ns) {
        record_timeout(status, bar, parity);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled load of one box into shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// 4-D tiled reduce-add of a shared-memory box into global memory (fp32 add in L2).
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2,
                                                  int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's committed bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// All but this thread's N most recently committed bulk groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_but() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
// This thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Named barrier over N threads.  The non-aligned form: threads of one warp may arrive at
// different times (one lane finishing a wait the others do not take part in), which the
// aligned bar.sync does not allow.
template <int ID, int N>
__device__ __forceinline__ void named_bar() {
  asm volatile("barrier.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, f32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Warp-issued forms: every lane of a converged warp executes the call with the same
// (warp-uniform) operands and one lane, chosen by elect.sync, issues the instruction.  Issuing
// from a converged warp keeps the descriptors in uniform registers, so a stream of MMAs costs
// a few instructions each and the tensor pipe is never starved by its own issue.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
// Descriptor of the operand `bytes` further on in shared memory (the start-address field holds
// address >> 4 and shared memory stays below 2^18 bytes, so the field never carries over).
__host__ __device__ constexpr uint64_t desc_at(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }
// A bounded wait taken by a whole warp: every lane returns the same verdict.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned *status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t), columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (tcgen05 format:
// start >> 4 in [0,14), leading byte offset >> 4 in [16,30), stride byte offset >> 4 in
// [32,46), version 1 in [46,48), base offset 0, swizzle mode 2 (128 B) in [61,64)).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The same for an operand without swizzling (swizzle mode 0), K-major: core matrices of
// 8 rows x 16 bytes, lbo_bytes apart along K and sbo_bytes apart along M / N.
__device__ __forceinline__ uint64_t plain_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and f32 accumulation.
// b_mn_major: B operand stored with its N dimension contiguous (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)   // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 1/d for d in [1, 2] on the FMA pipe (keeps the MUFU free for the exponentials):
// Newton-Raphson r <- r (2 - d r) from the linear minimax start 24/17 - 8/17 d (the classic
// 48/17 - 32/17 x estimate on [1/2, 1], rescaled), whose relative error 1/17 squares to
// ~3.5e-3 and then ~1.2e-5 after the two steps.
__device__ __forceinline__ float rcp_1to2(float d) {
  float r = fmaf(d, -0.47058823529411764f, 1.4117647058823530f);
  float e = fmaf(-d, r, 1.f);
  r = fmaf(r, e, r);
  e = fmaf(-d, r, 1.f);
  return fmaf(r, e, r);
}
// Packed pairs of fp32 (sm_100 family f32x2 arithmetic): one instruction for two lanes of
// element-wise work.  A pair lives in a 64-bit register (low word = first element).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_splat(float a) { return f2_pack(a, a); }

// r = 1 / (1 + 2^x) for a pair of x, on the FMA pipe apart from the one ex2 per element, so
// that the soft-cap costs the special-function unit one operation instead of three (a rcp
// issues at half the ex2 rate).  x is clamped to 126 so that d = 1 + 2^x stays finite.  The
// reciprocal starts from a bit-level seed -- the constant 0x7EF311C0 minus the bits of d
// negates the exponent and linearly approximates 1 / mantissa (minimax over a binade, found
// by a numerical search: max relative error 5.1 %) -- and two Newton-Raphson steps
// r <- r + r (1 - d r) square that error twice, to 6.5e-6 (always from below).  With
// t = cap (1 - 2 r) the logit error is at most 2 cap r 6.5e-6: vanishing for the largest
// logits (r -> 0), largest for the smallest (r -> 1, where P is negligible).
// Also returns e = 2^x (clamped like x), with which 1 - r = e r holds without cancellation.
__device__ __forceinline__ uint64_t f2_sigmoid2_neg(uint64_t x2, uint64_t &e2) {
  float xa, xb;
  f2_unpack(x2, xa, xb);
  const uint64_t m1 = f2_splat(-1.f), one = f2_splat(1.f);
  e2 = f2_pack(ex2_approx(fminf(xa, 126.f)), ex2_approx(fminf(xb, 126.f)));
  const uint64_t nd = f2_fma(e2, m1, m1);
  float na, nb;
  f2_unpack(nd, na, nb);  // -d: its bits are those of d plus the sign bit, folded into the constant
  uint64_t r = f2_pack(__uint_as_float(0xFEF311C0u - __float_as_uint(na)), __uint_as_float(0xFEF311C0u - __float_as_uint(nb)));
  r = f2_fma(r, f2_fma(nd, r, one), r);
  r = f2_fma(r, f2_fma(nd, r, one), r);
  return r;
}
__device__ __forceinline__ uint64_t f2_sigmoid2_neg(uint64_t x2) {
  uint64_t e2;
  return f2_sigmoid2_neg(x2, e2);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace tc

// Host: encode a 4-D bf16 tensor map (d, s, h, b) with a [64, box_rows, 1, 1] box and
// 128-byte swizzle.  Returns false if the driver entry point is unavailable or rejects it.
bool make_tmap_bshd(CUtensorMap *m, const void *base, int D, int S, int H, int B, long long stride_s,
                    long long stride_h, long long stride_b, int box_rows);

// Host: 4-D fp32 tensor map over a dense [B, S, H, D] array with a [box_d, box_rows, 1, 1]
// box, 128-byte swizzle or none (for bulk reduce-adds into the dQ accumulator).
bool make_tmap_f32_bshd(CUtensorMap *m, const void *base, int D, int S, int H, int B, int box_d, int box_rows,
                        bool swizzle128);

}  // namespace attn
