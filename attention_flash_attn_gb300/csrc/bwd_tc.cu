// bwd_tc.cu -- tcgen05 tensor-core backward for bf16, D in {64, 128, 256}.
//
// One CTA owns one 128-key tile of one (batch, kv head).  K and V stay in shared memory; the
// CTA walks the query heads of its GQA group and the query steps (BQ rows) that can see the
// tile, and accumulates dV and dK for its keys in tensor memory:
//
//   S^T  = K Q^T,  dP^T = V dO^T            (M = 128 keys, N = BQ; TMEM)
//   softmax warps (key = TMEM lane; two warps per lane quarter split the BQ columns):
//       t = cap*tanh(u/cap), mask, P = exp(t - LSE), dS = P (dP - D) (1 - tanh^2) * scale
//       -> P^T (bf16) into TMEM, dS^T (bf16, 128-byte swizzled) into shared memory
//   dV += P^T dO  (A = P^T from TMEM),  dK += dS^T Q  (A = dS^T from shared memory)
//   dQ  = dS K  (or dQ^T = K^T dS^T)  -> TMEM -> staged in shared memory -> TMA bulk
//       reduce-add into the fp32 dQ accumulator.
//
// The cap's chain-rule factor is applied before dK and dQ are formed (tokamax soft-capping
// VJP page).  P is recomputed from the forward's LSE with the forward's score function.  Each
// query step's Q, dO, LSE*log2(e) and D arrive together by TMA / bulk copy.  In the one-pass
// form (head dim 64 / 128) D arrives as -D split into bf16 parts and a K = 16 MMA against a
// tile of ones starts the dP^T accumulator at -D: every softmax thread would otherwise read
// each query's D from shared memory (a broadcast load that still costs the LSU several
// wavefronts), and subtract it.
//
// Head dim 256: dK and dV fill all 512 TMEM columns, so the CTA runs two passes over its
// query steps -- dV first, then dK and dQ (S^T recomputed).  V is not needed in the dV pass, so
// its shared-memory slot doubles as a second Q/dO stage there.  For the dK pass V moves into
// tensor memory (the A operand of dP^T = V dO^T), S^T and dP^T share one score buffer and dQ^T
// is produced one 128-row half at a time.  The dV-pass stages become two Q tile slots (Q_i
// resident from its S^T to its dK) and one dO slot, read by one MMA warp alone, and the rest
// of the second stage holds a second dS^T buffer and more dQ staging.  dK of a step is issued
// right after S^T of the next, and the softmax warps form P f from S^T before dP^T is in.
//
// Warps: 0..7 softmax / dS, 8 TMA producer, 9 MMA issuer + TMEM owner, 10 second MMA issuer
// (the MMAs that consume P and dS while warp 9 issues S^T / dP^T), 12..15 dQ drain.
// Every mbarrier is waited on phase by phase by each of its waiters: a parity wait cannot
// tell a phase from the one two later, so no waiter may skip one or fall two behind.
// Every wait is bounded (tc_common.cuh); named barriers are only used where every
// participating thread is guaranteed to arrive.
#include "bwd_score.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;
using namespace bwd_score;

constexpr int kBK = 128;  // keys per CTA
constexpr int kThreads = 512;
// Warpgroups: 0-1 softmax / dS (warps 0..7), 2 producers and MMA issuers (8 TMA, 9 front MMA
// and TMEM owner, 10 back MMA, 11 idle), 3 dQ drain (12..15).  Registers are moved from the
// producers and the drain to the softmax warpgroups (setmaxnreg): the element-wise loops need
// many values in flight to keep the MUFU busy.  128 threads x (176 + 176 + 72 + 80) stays
// within the 512 x 128 registers the CTA is launched with.
constexpr int kRegSoftmax = 176, kRegProducer = 72, kRegDrain = 80;
constexpr int kSoftmaxThreads = 256;
constexpr int kDrainThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int D_, int BQ_, bool DQT_, bool TWO_, int NS_>
struct BwdCfg {
  static constexpr int D = D_, BQ = BQ_, NS = NS_;
  static constexpr bool DQT = DQT_, TWO = TWO_;
  static constexpr int KCH = D / 64;
  static constexpr int KV_BYTES = kBK * D * 2;
  static constexpr int QT_BYTES = BQ * D * 2;
  static constexpr int SLOT_BYTES = 2 * QT_BYTES;  // Q, then dO
  static constexpr int NSLOT = TWO ? 2 : NS;       // two-pass: slot 1 is V's space (dV pass only)
  static constexpr int DS_BYTES = kBK * BQ * 2;
  static constexpr int DQS_BYTES = 16384;          // one bulk reduce box of fp32 dQ
  // Fused form: dP^T starts at -D.  One K = 16 MMA of a tile of ones against the step's -D,
  // split into three bf16 parts per query, fills the dP^T columns before the dP^T MMAs
  // accumulate onto them, so the softmax warps form dS = P f (dP - D) without reading D.
  // Both tiles use the no-swizzle K-major layout (8-row x 16-byte core matrices); per slot the
  // -D parts are [BQ rows x 8] bf16 (k = 0..7), followed by the zeros of k = 8..15.  They sit
  // below the K / V tiles.
  static constexpr bool FOLD = !TWO;
  static constexpr int ONES_BYTES = FOLD ? 4096 : 0;
  static constexpr int DSP_BYTES = FOLD ? BQ * 32 : 0;
  static constexpr int OFF_ONES = 0;
  static constexpr int OFF_DSP = OFF_ONES + ONES_BYTES;
  static constexpr int OFF_K = (ONES_BYTES + NSLOT * DSP_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_SLOT0 = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_DS = OFF_SLOT0 + NS * SLOT_BYTES;
  static constexpr int OFF_DQS = OFF_DS + DS_BYTES;
  static constexpr int OFF_LD = OFF_DQS + DQS_BYTES;  // per slot: LSE*log2e [BQ], D [BQ] (D unused in the fused form)
  static constexpr int OFF_BAR = OFF_LD + NSLOT * 2 * BQ * 4;
  static constexpr int NBAR = 12 + 2 * NSLOT + (TWO ? 23 : 0);  // + dQ half-1 release, dO hand-over, dS buffers
  // Two-pass form, dK pass: the dV pass's second dO stage holds the second dS^T buffer and two
  // more dQ staging boxes.
  static constexpr int OFF_DS1 = OFF_V + QT_BYTES;
  static constexpr int OFF_DQS2 = OFF_DS1 + DS_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  // TMEM columns
  static constexpr int TM_DV = 0;
  static constexpr int TM_DK = TWO ? 0 : D;
  static constexpr int TM_S = TWO ? 256 : 2 * D;
  static constexpr int TM_DP = TM_S + BQ;
  // Two-pass form: P lives in the dQ columns, idle during the dV pass.
  static constexpr int TM_P = TWO ? 384 : TM_DP + BQ;
  static constexpr int TM_DQ = TWO ? 384 : TM_P + BQ / 2;
  // Two-pass form, dK pass: V (bf16 pairs, the A operand of dP^T), one score buffer shared by
  // S^T and then dP^T, and one 128-row half of dQ^T at a time.
  static constexpr int TM_V = 256, TM_SDP = 384, TM_DQH = 448;
  static constexpr int DQ_COLS = DQT ? (D / 128) * BQ : D;
  static_assert(TM_DQ + DQ_COLS <= 512, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(!TWO || SLOT_BYTES == KV_BYTES, "the V slot must hold one Q/dO stage");
  static_assert(!TWO || DS_BYTES + DQS_BYTES <= QT_BYTES, "second dS^T buffer and staging fit a dO stage");
  static_assert(!DQT || D % 128 == 0, "transposed dQ needs whole 128-row halves of D");
  static_assert(DQT || (BQ == 128 && D == 64), "row-major dQ is the D = 64, BQ = 128 form");
  static_assert(BQ % 64 == 0, "dS^T rows are whole 128-byte swizzle rows");
};

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int e = 0; e < N; ++e) asm volatile("" : "+r"(r[e]));
}

__device__ __forceinline__ uint4 pack8(const uint32_t *o, int v) {
  return make_uint4(pack_bf16(__uint_as_float(o[8 * v]), __uint_as_float(o[8 * v + 1])),
                    pack_bf16(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3])),
                    pack_bf16(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5])),
                    pack_bf16(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7])));
}

// Bias of this thread's key for the 32 queries q0 .. q0 + 31 of a chunk, as 16 bf16 pairs
// (query q0 + 2 e in the low half of pair e).  `col` points at the key's column of the head's
// [Sq, Sk] bias rows; rows past Sq read row Sq - 1 (their probabilities are zero).  A warp's
// 32 keys are consecutive, so each load instruction reads 64 contiguous bytes.
__device__ __forceinline__ void load_bias_col(uint32_t (&bq)[16], const unsigned short *col, int q0, int Sq,
                                              long long Sk) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int qa = min(q0 + 2 * e, Sq - 1), qb = min(q0 + 2 * e + 1, Sq - 1);
    bq[e] = (uint32_t)__ldg(col + qa * Sk) | ((uint32_t)__ldg(col + qb * Sk) << 16);
  }
}

// One 32-query chunk of a key row, every column treated as visible (masked columns are
// cleared afterwards by the fix-ups below, only on chunks that need it):
//   KIND 1: P, packed to bf16 pairs;  KIND 0: P and dS = P f (dP - D), both packed, from the
//   dP^T accumulator that started at -D.
//   BIAS: bq holds the chunk's bias pairs; with KIND 0, dU = P f (dP - D) of each visible
//   query (vis bit e) is also added into the dbias accumulator at dbc + e Sk.
template <bool CAP, bool FRCP, int KIND, bool BIAS = false>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&sr)[32], const uint32_t (&dr)[32], const float *lse2c,
                                          uint32_t (&pk)[16], uint32_t (&dk)[16], const BwdScore &k,
                                          const uint32_t *bq = nullptr, float *dbc = nullptr, long long Sk = 0,
                                          uint32_t vis = 0) {
  const uint64_t *l2 = reinterpret_cast<const uint64_t *>(lse2c);
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    uint64_t y, f;
    score_pair<CAP, FRCP, BIAS>(sr[2 * e2], sr[2 * e2 + 1], l2[e2], k, y, f, BIAS ? bias_pair(bq[e2]) : 0);
    const uint64_t p2 = ex2_pair(y);
    pk[e2] = bf16_pair(p2);
    if constexpr (KIND == 0) {
      const uint64_t dpd = f2_pack(__uint_as_float(dr[2 * e2]), __uint_as_float(dr[2 * e2 + 1]));
      const uint64_t du = f2_mul(f2_mul(p2, f), dpd);
      if constexpr (BIAS) {
        float a, b;
        f2_unpack(du, a, b);
        red_add_f32_if(dbc + (2 * e2) * Sk, a, (vis >> (2 * e2)) & 1u);
        red_add_f32_if(dbc + (2 * e2 + 1) * Sk, b, (vis >> (2 * e2 + 1)) & 1u);
        dk[e2] = bf16_pair(f2_mul(du, k.scale));
      } else {
        dk[e2] = bf16_pair(du);
      }
    }
  }
}

// The dK pass's chunk in two steps, so that the first runs before dP^T has been computed:
// (1) in place, the raw score -> P f;
template <bool CAP, bool FRCP, bool BIAS = false>
__device__ __forceinline__ void ds_first(uint32_t (&sr)[32], const float *lse2c, const BwdScore &k,
                                         const uint32_t *bq = nullptr) {
  const uint64_t *l2 = reinterpret_cast<const uint64_t *>(lse2c);
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    uint64_t y, f;
    score_pair<CAP, FRCP, BIAS>(sr[2 * e2], sr[2 * e2 + 1], l2[e2], k, y, f, BIAS ? bias_pair(bq[e2]) : 0);
    float a, b;
    f2_unpack(f2_mul(ex2_pair(y), f), a, b);
    sr[2 * e2] = __float_as_uint(a);
    sr[2 * e2 + 1] = __float_as_uint(b);
  }
}
// (2) dS = P f (dP - D), packed to bf16 pairs.  BIAS: P f came without the softmax scale;
// dU = P f (dP - D) of each visible query goes into the dbias accumulator first.
template <bool BIAS = false>
__device__ __forceinline__ void ds_second(const uint32_t (&pf)[32], const uint32_t (&dr)[32], const float *dvc,
                                          uint32_t (&dk)[16], uint64_t scale2 = 0, float *dbc = nullptr,
                                          long long Sk = 0, uint32_t vis = 0) {
  const uint64_t *d2 = reinterpret_cast<const uint64_t *>(dvc);
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    const uint64_t pf2 = f2_pack(__uint_as_float(pf[2 * e2]), __uint_as_float(pf[2 * e2 + 1]));
    const uint64_t dp = f2_pack(__uint_as_float(dr[2 * e2]), __uint_as_float(dr[2 * e2 + 1]));
    const uint64_t du = f2_mul(pf2, f2_sub(dp, d2[e2]));
    if constexpr (BIAS) {
      float a, b;
      f2_unpack(du, a, b);
      red_add_f32_if(dbc + (2 * e2) * Sk, a, (vis >> (2 * e2)) & 1u);
      red_add_f32_if(dbc + (2 * e2 + 1) * Sk, b, (vis >> (2 * e2 + 1)) & 1u);
      dk[e2] = bf16_pair(f2_mul(du, scale2));
    } else {
      dk[e2] = bf16_pair(du);
    }
  }
}

// Visibility of the 32 query columns qb .. qb + 31 for this thread's key: bit e is set when
// query qb + e lies in [lo, hi) and, with unsorted segment ids, shares the key's segment.
__device__ __forceinline__ uint32_t chunk_vis(int qb, int lo, int hi, bool pairwise, const int *segq, int sq,
                                              int sid) {
  const int a = max(lo - qb, 0), b = min(hi - qb, 32);
  if (a >= b) return 0u;
  uint32_t v = (b == 32 ? 0xffffffffu : ((1u << b) - 1u)) & ~((1u << a) - 1u);
  if (pairwise) {
    uint32_t same = 0u;
#pragma unroll 1
    for (int e = 0; e < 32; ++e) same |= (uint32_t)(__ldg(segq + min(qb + e, sq - 1)) == sid) << e;
    v &= same;
  }
  return v;
}
// Clear the hidden columns of a chunk: 32 fp32 values, or 16 bf16 pairs.
__device__ __forceinline__ void clear_hidden(uint32_t (&x)[32], uint32_t vis) {
#pragma unroll
  for (int e = 0; e < 32; ++e) x[e] = ((vis >> e) & 1u) ? x[e] : 0u;
}
__device__ __forceinline__ void clear_hidden(uint32_t (&x)[16], uint32_t vis) {
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2)
    x[e2] &= (((vis >> (2 * e2)) & 1u) ? 0x0000ffffu : 0u) | (((vis >> (2 * e2 + 1)) & 1u) ? 0xffff0000u : 0u);
}

// GM: the group-major grid order (chosen on the host, below).
template <class C, bool CAP, bool BIAS, bool GM>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmDQ, const Params p) {
  constexpr int D = C::D, BQ = C::BQ, NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *misc_i = reinterpret_cast<int *>(smem + C::OFF_MISC);
  {  // A wait elsewhere already gave up: do nothing (decided once for the whole CTA).
    if (threadIdx.x == 0) misc_i[12] = (status_peek(p.status) & kStatusWaitTimeout) ? 1 : 0;
    __syncthreads();
    if (misc_i[12]) return;
  }

  // One-dimensional grid, heaviest tiles first so that the last wave holds the light ones.
  // With segments the order is the mask metadata's longest-first work list of (batch, key
  // tile) pairs, every kv head of a pair adjacent; otherwise the key tile varies slowest,
  // earliest (seen by the most queries under causal masks) first -- or, for query ranges of
  // 16k rows and more, the (batch, kv head) group varies slowest.  Measured on the same box:
  // long causal 32k backward 658 -> 718 TFLOP/s and long non-causal 16k 841 -> 873 group-major,
  // but the windowed 8k workload 824 -> 642 and the sink workload 685 -> 548: there a group's
  // key tiles in flight together reduce into the same dQ rows at once.
  const int nkt = (p.Sk + kBK - 1) / kBK;
  int kt, g, b;
  if (p.korder) {
    const int2 o = p.korder[blockIdx.x / (unsigned)p.Hkv];
    b = o.x;
    kt = o.y;
    g = (int)(blockIdx.x % (unsigned)p.Hkv);
  } else if (GM) {
    // Long query ranges: the key tiles of one (batch, kv head) run together, earliest first, so
    // the CTAs in flight read that group's Q / dO rows from L2 at staggered starts.
    const int gb = (int)(blockIdx.x / (unsigned)nkt);
    kt = (int)(blockIdx.x % (unsigned)nkt);
    g = gb % p.Hkv;
    b = gb / p.Hkv;
  } else {
    const int gb = (int)(blockIdx.x % (unsigned)(p.Hkv * p.B));
    kt = (int)(blockIdx.x / (unsigned)(p.Hkv * p.B));
    g = gb % p.Hkv;
    b = gb / p.Hkv;
  }
  const int k0 = kt * kBK, k1 = min(k0 + kBK, p.Sk) - 1;
  const int off = p.Sk - p.Sq;

  // Query rows that can see this key tile (uniform across the CTA).
  int qlo = 0, qhi = p.Sq;
  if (!p.koff) {  // per-sequence offsets: the tile ranges below carry the causal / window bounds
    if (p.causal) qlo = max(qlo, k0 - off);
    if (p.window > 0) qhi = min(qhi, k1 - off + p.window);
  }
  if (p.ktile) {  // the tile's class bounds from the mask metadata
    const int4 c = p.ktile[(size_t)b * nkt + kt];
    qlo = max(qlo, c.x);
    qhi = min(qhi, c.y);
  }
  const int s0 = qlo / BQ;
  const int nq = (qlo < qhi) ? (qhi + BQ - 1) / BQ - s0 : 0;  // query steps per head
  const int nper = nq * p.G;                                   // steps per pass
  const int nsteps = C::TWO ? 2 * nper : nper;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t kv_full = bar0, v_full = bar0 + 8u;
  const uint32_t s_full = bar0 + 16u, p_ready = bar0 + 24u, mma_done = bar0 + 32u;
  const uint32_t dq_full = bar0 + 40u, acc_free = bar0 + 56u, fin_done = bar0 + 64u;
  // dq_empty(m): the drain has copied half m (d rows 128 m .. 128 m + 127 of dQ^T) out of TMEM.
  auto dq_empty = [&](int m) { return m == 0 ? bar0 + 48u : bar0 + 8u * (C::NBAR - 1); };
  // Two-pass form: the dV pass's first dO stage is free for the ring.  Lane 1, which waits on
  // that stage's releases in order, hands it to lane 0 through this single-phase barrier (a
  // waiter that has not seen a barrier's earlier phases could mistake one for the next).
  const uint32_t do0_free = bar0 + 8u * (C::NBAR - 2);
  // Two-pass form, dK pass: dS^T is double-buffered (buffer i & 1 for step i).  p_ready_b(x):
  // the softmax has stored buffer x; dsb_done(x): dK and dQ of the step that read buffer x have
  // completed.  Per-buffer barriers keep a barrier's phases two steps apart.
  auto p_ready_b = [&](int x) { return bar0 + 8u * (C::NBAR - 7 + x); };
  auto dsb_done = [&](int x) { return bar0 + 8u * (C::NBAR - 5 + x); };
  const uint32_t sdp_free = bar0 + 72u;  // S^T / dP^T copied out of TMEM (256 arrivals)
  // Q/dO stages; in the two-pass form these are the Q ring, and do_full / do_empty the dO ring.
  auto qdo_full = [&](int s) { return bar0 + 8u * (10 + s); };
  auto qdo_empty = [&](int s) { return bar0 + 8u * (10 + C::NSLOT + s); };
  auto do_full = [&](int s) { return bar0 + 8u * (10 + 2 * C::NSLOT + s); };
  auto do_empty = [&](int s) { return bar0 + 8u * (12 + 2 * C::NSLOT + s); };
  // Two-pass form: LSE*log2e / D of step j in their own two-deep ring (index j & 1), filled by
  // the Q lane and released by the softmax warps once they have read it.
  auto ld_full = [&](int x) { return bar0 + 8u * (14 + 2 * C::NSLOT + x); };
  auto ld_empty = [&](int x) { return bar0 + 8u * (16 + 2 * C::NSLOT + x); };
  // Two-pass form, dK pass: V moves to tensor memory, and the dV pass's stages become two Q tile
  // slots (Q_i in slot i & 1, resident from its S^T to its dK after the softmax of step i) and
  // one dO slot (released by dP^T_i); the second dO stage holds the second dS^T buffer and more
  // dQ staging.  Each slot has one full and one empty barrier, so the MMA warp waits and
  // commits once per tile (a commit between MMA groups costs the tensor pipe a drain).
  auto ring_full = [&](int r) { return bar0 + 8u * (18 + 2 * C::NSLOT + r); };
  auto ring_empty = [&](int r) { return bar0 + 8u * (22 + 2 * C::NSLOT + r); };
  const uint32_t dp_full = bar0 + 8u * (26 + 2 * C::NSLOT);  // dP^T of a dK-pass step is in TMEM
  const uint32_t dp_free = bar0 + 8u * (27 + 2 * C::NSLOT);  // ... and has been copied out (256)
  // slots 0, 1 (Q): the first stage's Q and dO; slot 2 (dO): the second stage's Q
  auto ring_addr = [&](int r) -> uint32_t {
    return sbase + (r < 2 ? C::OFF_SLOT0 + r * C::QT_BYTES : C::OFF_V);
  };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *red = misc_i + 4;  // [8]

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(v_full, C::TWO ? kSoftmaxThreads : 1);  // two-pass: every softmax thread stores its part of V
    mbar_init(s_full, 1);
    mbar_init(p_ready, kSoftmaxThreads);
    mbar_init(mma_done, C::TWO ? 2 : 1);  // two-pass: dV / dQ (back warp) and dK (front warp)
    mbar_init(do0_free, 1);
    if (C::TWO) {
      for (int x = 0; x < 2; ++x) {
        mbar_init(p_ready_b(x), kSoftmaxThreads);
        mbar_init(dsb_done(x), 2);  // dK (front warp) and dQ (back warp)
      }
    }
    mbar_init(dq_full, 1);
    mbar_init(dq_empty(0), kDrainThreads);  // every drain thread has read (its half of) the dQ tile
    mbar_init(dq_empty(1), kDrainThreads);
    mbar_init(acc_free, kSoftmaxThreads);
    mbar_init(fin_done, 2);  // both MMA warps have finished
    mbar_init(sdp_free, kSoftmaxThreads);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(qdo_full(s), 1);
      mbar_init(qdo_empty(s), 1);
      if (C::TWO) {
        mbar_init(do_full(s), 1);
        mbar_init(do_empty(s), 1);
        mbar_init(ld_full(s), 1);
        mbar_init(ld_empty(s), kSoftmaxThreads);
      }
    }
    if (C::TWO) {
      for (int r = 0; r < 3; ++r) {
        mbar_init(ring_full(r), 1);
        mbar_init(ring_empty(r), 1);
      }
      mbar_init(dp_full, 1);
      mbar_init(dp_free, kSoftmaxThreads);
    }
    fence_barrier_init();
  }
  if constexpr (C::FOLD) {
    // The tile of ones (bf16 1.0) and the zero half of each -D tile, written once: the TMA
    // only ever writes the -D half.
    for (int i = threadIdx.x; i < C::ONES_BYTES / 16; i += kThreads)
      reinterpret_cast<uint4 *>(smem + C::OFF_ONES)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    for (int i = threadIdx.x; i < C::NSLOT * BQ; i += kThreads)
      reinterpret_cast<uint4 *>(smem + C::OFF_DSP + (i / BQ) * C::DSP_BYTES + BQ * 16)[i % BQ] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();  // visible to the tensor cores after the barrier below
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // step j -> (head, first query row, pass kind: 0 fused, 1 dV pass, 2 dK+dQ pass),
  // its Q/dO slot and that slot's use count (for mbarrier phases).
  auto step_h = [&](int j) { return g * p.G + (j % nper) / nq; };
  auto step_q0 = [&](int j) { return (s0 + (j % nper) % nq) * BQ; };
  auto step_kind = [&](int j) { return C::TWO ? (j < nper ? 1 : 2) : 0; };
  auto slot_of = [&](int j) { return C::TWO ? (j < nper ? (j & 1) : 0) : (j % NS); };
  auto use_of = [&](int j) { return C::TWO ? (j < nper ? (j >> 1) : ((nper + 1) >> 1) + (j - nper)) : (j / NS); };
  // Q tile of slot s; its dO tile is QT_BYTES further (fused) -- in the two-pass form the Q
  // ring is {R0, R2} and the dO ring {R1, R3}, R2/R3 being V's space during the dV pass.
  auto slot_addr = [&](int s) -> uint32_t {
    return (C::TWO && s == 1) ? sbase + C::OFF_V : sbase + C::OFF_SLOT0 + s * C::SLOT_BYTES;
  };
  auto do_addr = [&](int s) -> uint32_t { return slot_addr(s) + C::QT_BYTES; };
  auto ld_addr = [&](int s) { return reinterpret_cast<const float *>(smem + C::OFF_LD + s * 2 * BQ * 4); };

  // Each warpgroup sets its register budget as the first statement of its own branch, so
  // the code of a role is only reachable under that role's budget.
  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
    // ------------------------------------------------------------ softmax / dS warps
    const int wq = warp & 3;
    const int half = warp >> 2;  // which half of the BQ query columns
    const int r = wq * 32 + lane;      // key row within the tile == TMEM lane
    const int k = k0 + r;
    const bool key_ok = k < p.Sk;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);

    // Query interval [lo, hi) that sees this key; keys past Sk see nothing.
    int lo = 0, hi = p.Sq;
    const int koff = key_ok ? key_off(p, k) : off;
    if (p.causal) lo = max(lo, k - koff);
    if (p.window > 0) hi = min(hi, k - koff + p.window);
    bool seg_pairwise = false;
    int sid = 0;
    const int *segq = nullptr;
    if (p.seg_q && key_ok) {
      if (p.seg_mono[b]) {  // sorted ids: the metadata's interval for this key (its segment's run)
        const int2 x = __ldg(p.krun + (size_t)b * p.Sk + k);
        lo = max(lo, x.x);
        hi = min(hi, x.y);
      } else {
        sid = __ldg(p.seg_k + (size_t)b * p.Sk + k);
        segq = p.seg_q + (size_t)b * p.Sq;
        seg_pairwise = true;
      }
    }
    if (!key_ok) {
      lo = p.Sq;
      hi = 0;
    }
    // Queries that see every key of the tile, [cta_lo, cta_hi): query steps inside need no
    // mask.  The mask metadata carries them (the tile class); otherwise the keys' intervals are
    // intersected here.
    int cta_lo, cta_hi;
    if (p.ktile) {
      const int4 c = p.ktile[(size_t)b * nkt + kt];
      cta_lo = c.z;
      cta_hi = c.w;
    } else {
      if (half == 0) {
        int mlo = __reduce_max_sync(0xffffffffu, lo);
        int mhi = __reduce_min_sync(0xffffffffu, hi);
        if (lane == 0) {
          red[wq] = mlo;
          red[4 + wq] = mhi;
        }
      }
      named_bar<1, kSoftmaxThreads>();
      cta_lo = max(max(red[0], red[1]), max(red[2], red[3]));
      cta_hi = min(min(red[4], red[5]), min(red[6], red[7]));
    }
    const bool any_pairwise = p.seg_q != nullptr && !p.seg_mono[b];

    const BwdScore ks(p.scale, p.inv_cap, p.cap);
    uint8_t *ds_row = smem + C::OFF_DS + r * 128;
    bool ok = true;
    // Bias: this key's column of the [Sq, Sk] rows of each query head (a key past Sk reads
    // the last column; its queries are never visible), and the same column of the fp32 dbias
    // accumulator, whose broadcast dimensions have extent 1.
    const int kc = key_ok ? k : p.Sk - 1;
    const unsigned short *bias_b =
        BIAS ? static_cast<const unsigned short *>(p.bias) + (size_t)b * p.bias_sb + kc : nullptr;
    float *dbias_b = BIAS ? p.dbias_acc + (size_t)(p.bias_B == 1 ? 0 : b) * p.bias_H * p.Sq * p.Sk + kc : nullptr;

    for (int j = 0; j < nsteps && ok; ++j) {
      const int kind = step_kind(j), q0 = step_q0(j), s = slot_of(j);
      constexpr int NCH = BQ / 64;  // 32-column chunks per thread and step
      uint32_t bq[NCH][BIAS ? 16 : 1];
      const unsigned short *bcol = nullptr;
      float *dbcol = nullptr;
      if constexpr (BIAS) {  // the step's bias, in flight while S^T is computed
        const int h = step_h(j);
        bcol = bias_b + (size_t)h * p.bias_sh;
        dbcol = dbias_b + (size_t)(p.bias_H == 1 ? 0 : h) * p.Sq * p.Sk;
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) load_bias_col(bq[cc], bcol, q0 + (half * NCH + cc) * 32, p.Sq, p.Sk);
      }
      if (!mbar_wait(s_full, j & 1, p.status)) { ok = false; break; }
      if (C::TWO) {
        if (!mbar_wait(ld_full(j & 1), (j >> 1) & 1, p.status)) { ok = false; break; }
      } else {
        if (!mbar_wait(qdo_full(s), use_of(j) & 1, p.status)) { ok = false; break; }
      }
      tc_fence_after();
      const float *lse2 = ld_addr(C::TWO ? (j & 1) : s);
      const float *dvv = lse2 + BQ;
      const bool full = !any_pairwise && q0 >= cta_lo && q0 + BQ <= cta_hi;

      // P and dS of this thread's columns are formed in registers while the previous
      // step's dV / dK / dQ MMAs still read the P^T and dS^T buffers (and, once S^T / dP^T
      // are copied out, while the next step's S^T / dP^T are computed) ...
      uint32_t pk[NCH][16], dk[NCH][16];
      if (C::TWO && kind == 2) {
        // dK pass: P f from S^T first, then dP^T (computed meanwhile) for dS.
        uint32_t pf[NCH][32];
        uint32_t visc[NCH];
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int c = half * NCH + cc;
          tmem_ld32(lane_addr + C::TM_SDP + c * 32, pf[cc]);
          tmem_wait_ld();
          reg_fence(pf[cc]);
          if (cc == NCH - 1) {
            tc_fence_before();
            mbar_arrive(sdp_free);
          }
          ds_first<CAP, false, BIAS>(pf[cc], lse2 + c * 32, ks, bq[cc]);
          visc[cc] = full ? 0xffffffffu : chunk_vis(q0 + c * 32, lo, hi, seg_pairwise, segq, p.Sq, sid);
          if (!full) clear_hidden(pf[cc], visc[cc]);
        }
        if (!mbar_wait(dp_full, (j - nper) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int c = half * NCH + cc;
          uint32_t dr[32];
          tmem_ld32(lane_addr + C::TM_SDP + c * 32, dr);
          tmem_wait_ld();
          reg_fence(dr);
          if (cc == NCH - 1) {
            tc_fence_before();
            mbar_arrive(dp_free);
          }
          ds_second<BIAS>(pf[cc], dr, dvv + c * 32, dk[cc], ks.scale, BIAS ? dbcol + (size_t)(q0 + c * 32) * p.Sk : nullptr,
                          p.Sk, visc[cc]);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int c = half * NCH + cc;  // 32-column chunk of this step
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_addr + C::TM_S + c * 32, sr);
          if constexpr (!C::TWO) tmem_ld32(lane_addr + C::TM_DP + c * 32, dr);
          tmem_wait_ld();
          reg_fence(sr);
          if constexpr (!C::TWO) reg_fence(dr);
          if (cc == NCH - 1) {
            tc_fence_before();
            mbar_arrive(sdp_free);
          }
          if constexpr (BIAS) {
            const uint32_t vis = full ? 0xffffffffu : chunk_vis(q0 + c * 32, lo, hi, seg_pairwise, segq, p.Sq, sid);
            bwd_chunk<CAP, true, C::TWO ? 1 : 0, true>(sr, dr, lse2 + c * 32, pk[cc], dk[cc], ks, bq[cc],
                                                       dbcol + (size_t)(q0 + c * 32) * p.Sk, p.Sk, vis);
            if (!full) {
              clear_hidden(pk[cc], vis);
              if (!C::TWO) clear_hidden(dk[cc], vis);
            }
          } else {
            bwd_chunk<CAP, true, C::TWO ? 1 : 0>(sr, dr, lse2 + c * 32, pk[cc], dk[cc], ks);
            if (!full) {
              const uint32_t vis = chunk_vis(q0 + c * 32, lo, hi, seg_pairwise, segq, p.Sq, sid);
              clear_hidden(pk[cc], vis);
              if (!C::TWO) clear_hidden(dk[cc], vis);
            }
          }
        }
      }
      if (C::TWO) mbar_arrive(ld_empty(j & 1));  // LSE / D of this step have been read
      // ... and stored once those MMAs are done with the buffers (the dK pass double-buffers
      // dS^T: buffer i & 1 was last read by dK / dQ of step i - 2).
      const int ib = j - nper;
      if (C::TWO && kind == 2) {
        if (ib >= 2 && !mbar_wait(dsb_done(ib & 1), ((ib >> 1) - 1) & 1, p.status)) { ok = false; break; }
      } else if (j >= 1 && !mbar_wait(mma_done, (j - 1) & 1, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t *ds_buf = (C::TWO && kind == 2 && (ib & 1)) ? smem + C::OFF_DS1 + r * 128 : ds_row;
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = half * NCH + cc;
        if (kind != 2) tmem_st16(lane_addr + C::TM_P + c * 16, pk[cc]);
        if (kind != 1) {
          // 32 queries = 64 bytes = four 16-byte units of this row, swizzled by (row & 7)
          uint8_t *chunk = ds_buf + (c >> 1) * (kBK * 128);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int unit = ((c & 1) * 4 + v) ^ (r & 7);
            *reinterpret_cast<uint4 *>(chunk + unit * 16) =
                make_uint4(dk[cc][4 * v], dk[cc][4 * v + 1], dk[cc][4 * v + 2], dk[cc][4 * v + 3]);
          }
        }
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive((C::TWO && kind == 2) ? p_ready_b(ib & 1) : p_ready);

      if (C::TWO && j == nper - 1) {
        // End of the dV pass: store dV (this warp's half of the columns), then hand the
        // accumulator over to dK.
        if (!mbar_wait(mma_done, j & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.dV) + (((size_t)b * p.Sk + k) * p.Hkv + g) * D;
#pragma unroll 1
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          uint32_t o[32];
          tmem_ld32(lane_addr + C::TM_DV + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (key_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v) reinterpret_cast<uint4 *>(dst + c * 32)[v] = pack8(o, v);
          }
        }
        tc_fence_before();
        mbar_arrive(acc_free);
        // V into tensor memory for the dK pass (A operand of dP^T): this thread's key row,
        // its half of D as bf16 pairs (the last dV-pass S^T, which lived there, is read).
        const uint4 *vsrc = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.v) + (size_t)b * p.v_sb +
                                                            (size_t)(key_ok ? k : 0) * p.v_ss + (size_t)g * p.v_sh +
                                                            half * (D / 2));
#pragma unroll 1
        for (int c = 0; c < D / 128; ++c) {
          uint32_t vv[32];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = key_ok ? __ldg(vsrc + c * 8 + v) : make_uint4(0, 0, 0, 0);
            vv[4 * v] = x.x;
            vv[4 * v + 1] = x.y;
            vv[4 * v + 2] = x.z;
            vv[4 * v + 3] = x.w;
          }
          tmem_st32(lane_addr + C::TM_V + half * (D / 4) + c * 32, vv);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(v_full);
      }
    }

    // Epilogue: dK (and dV in the single-pass form), this warp's half of the columns.
    if (ok && nsteps > 0) {
      ok = mbar_wait(fin_done, 0, p.status);
      tc_fence_after();
    }
    const bool have = nsteps > 0;
    for (int which = C::TWO ? 1 : 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? C::TM_DV : C::TM_DK;
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(which == 0 ? p.dV : p.dK) +
                           (((size_t)b * p.Sk + k) * p.Hkv + g) * D;
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t o[32];
        if (have) {
          tmem_ld32(lane_addr + col + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (key_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) reinterpret_cast<uint4 *>(dst + c * 32)[v] = pack8(o, v);
        }
      }
    }
    if (C::TWO && nsteps == 0 && key_ok) {  // no query sees these keys: dV is zero too
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dV) +
                                             (((size_t)b * p.Sk + k) * p.Hkv + g) * D);
      for (int v = half * (D / 16); v < (half + 1) * (D / 16); ++v) dst[v] = make_uint4(0, 0, 0, 0);
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegProducer));
    if (warp == 8 && C::TWO) {
      // ------------------------------------------------------------ TMA producers (two-pass)
      // dV pass: lane 0 loads K, the Q ring and the LSE / D ring, lane 1 the dO ring.  dK pass:
      // lane 0 alone fills the tile ring (Q_i, dO_i) and the LSE / D ring; lane 1 hands the dV
      // pass's dO stages over.  Every ring has one loader at a time and its waits run in phase
      // order.
      const int u_last0 = ((nper + 1) >> 1) - 1;  // last dV-pass use of stage 0
      const int u_last1 = (nper >> 1) - 1;        // ... and of stage 1
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        mbar_arrive_expect_tx(kv_full, C::KV_BYTES);
  #pragma unroll
        for (int c = 0; c < C::KCH; ++c) tma_load_4d(sbase + C::OFF_K + c * (kBK * 128), &tmK, kv_full, c * 64, k0, g, b);
        // One Q or dO tile (rows q0 .. q0 + BQ - 1) into ring slot r for its use u.  The first
        // use of a slot waits for the dV pass's last use of that region: the first stage's Q
        // (slot 0) and dO (slot 1, handed over by lane 1), the second stage's Q (slot 2).
        auto ring_load = [&](const CUtensorMap *tm, int r, int u, int q0, int h) -> bool {
          bool ok = true;
          if (u >= 1)
            ok = mbar_wait(ring_empty(r), (u - 1) & 1, p.status);
          else if (r == 0)
            ok = mbar_wait(qdo_empty(0), u_last0 & 1, p.status);
          else if (r == 1)
            ok = mbar_wait(do0_free, 0, p.status);
          else
            ok = u_last1 < 0 || mbar_wait(qdo_empty(1), u_last1 & 1, p.status);
          if (!ok) return false;
          mbar_arrive_expect_tx(ring_full(r), C::QT_BYTES);
  #pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(ring_addr(r) + c * (BQ * 128), tm, ring_full(r), c * 64, q0, h, b);
          return true;
        };
        for (int j = 0; j < nsteps; ++j) {
          {  // LSE / D of step j first: the softmax needs them with S^T_j
            const int x = j & 1, h = step_h(j), q0 = step_q0(j);
            if (j >= 2 && !mbar_wait(ld_empty(x), ((j >> 1) - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(ld_full(x), 2 * BQ * 4);
            const size_t row = ((size_t)b * p.Hq + h) * p.sq_pad + q0;
            const uint32_t lda = sbase + C::OFF_LD + x * 2 * BQ * 4;
            bulk_g2s(lda, p.lse2p + row, BQ * 4, ld_full(x));
            bulk_g2s(lda + BQ * 4, p.Dvec + row, BQ * 4, ld_full(x));
          }
          if (j < nper) {
            const int s = slot_of(j), u = use_of(j);
            if (u >= 1 && !mbar_wait(qdo_empty(s), (u - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(qdo_full(s), C::QT_BYTES);
  #pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(slot_addr(s) + c * (BQ * 128), &tmQ, qdo_full(s), c * 64, step_q0(j), step_h(j), b);
          } else {
            // Q_i (slot i & 1) for S^T and dK, dO_i (slot 2) for dP^T
            const int i = j - nper, h = step_h(j), q0 = step_q0(j);
            if (!ring_load(&tmQ, i & 1, i >> 1, q0, h) || !ring_load(&tmdO, 2, i, q0, h)) break;
          }
        }
      } else if (lane == 1) {
        tma_prefetch_desc(&tmdO);
        bool ok = true;
        for (int j = 0; j < nper; ++j) {
          const int s = slot_of(j), u = use_of(j);
          if (u >= 1 && !mbar_wait(do_empty(s), (u - 1) & 1, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(do_full(s), C::QT_BYTES);
  #pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(do_addr(s) + c * (BQ * 128), &tmdO, do_full(s), c * 64, step_q0(j), step_h(j), b);
        }
        // The first dO stage, once its last dV-pass use is released, becomes Q slot 1.  (The
        // second dO stage's new uses start after the dV pass's last MMAs have completed.)
        if (ok && nper > 0 && mbar_wait(do_empty(0), u_last0 & 1, p.status)) mbar_arrive(do0_free);
      }
    } else if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        mbar_arrive_expect_tx(kv_full, (C::TWO ? 1 : 2) * C::KV_BYTES);
  #pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_4d(sbase + C::OFF_K + c * (kBK * 128), &tmK, kv_full, c * 64, k0, g, b);
          if (!C::TWO) tma_load_4d(sbase + C::OFF_V + c * (kBK * 128), &tmV, kv_full, c * 64, k0, g, b);
        }
        for (int j = 0; j < nsteps; ++j) {
          if (C::TWO && j == nper) {
            // The dK pass needs V: wait until the dV pass has released V's slot, then load it.
            if (nper >= 2 && !mbar_wait(qdo_empty(1), ((nper >> 1) - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(v_full, C::KV_BYTES);
  #pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(sbase + C::OFF_V + c * (kBK * 128), &tmV, v_full, c * 64, k0, g, b);
          }
          const int s = slot_of(j), u = use_of(j);
          if (u >= 1 && !mbar_wait(qdo_empty(s), (u - 1) & 1, p.status)) break;
          const int h = step_h(j), q0 = step_q0(j);
          const uint32_t sa = slot_addr(s);
          mbar_arrive_expect_tx(qdo_full(s), 2 * C::QT_BYTES + BQ * 4 + BQ * 16);
  #pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_4d(sa + c * (BQ * 128), &tmQ, qdo_full(s), c * 64, q0, h, b);
            tma_load_4d(sa + C::QT_BYTES + c * (BQ * 128), &tmdO, qdo_full(s), c * 64, q0, h, b);
          }
          const size_t row = ((size_t)b * p.Hq + h) * p.sq_pad + q0;
          bulk_g2s(sbase + C::OFF_LD + s * 2 * BQ * 4, p.lse2p + row, BQ * 4, qdo_full(s));
          bulk_g2s(sbase + C::OFF_DSP + s * C::DSP_BYTES, p.dsplit + row, BQ * 16, qdo_full(s));
        }
      }
    } else if (warp == 9 || warp == 10) {
      // ------------------------------------------------------------ MMA issuers
      // Each issuing warp runs its loop with warp-uniform values and one elected lane issues
      // each MMA and commit; descriptors are built once per operand and advanced by constant
      // offsets.  Warp 9 issues the front MMAs (S^T, dP^T; in the dK pass also dK, so that it is
      // the only reader of the ring) and warp 10 the back ones (dV, dQ; in the fused form dV,
      // dK, dQ), so neither waits behind the other's queue.
      const bool back_warp = warp == 10;
      {
        constexpr uint32_t idST = idesc_bf16(kBK, BQ, false, false);  // S^T, dP^T
        constexpr uint32_t idKV = idesc_bf16(kBK, D, false, true);    // dV, dK
        constexpr uint32_t idKh = idesc_bf16(kBK, D / 2, false, true);  // one half of dK (two-pass)
        constexpr uint32_t idDQ = C::DQT ? idesc_bf16(128, BQ, true, true) : idesc_bf16(BQ, D, true, true);
        const uint64_t dK_k = sw128_desc(sbase + C::OFF_K, 16, 1024);          // K, K-major (A of S^T)
        const uint64_t dV_k = sw128_desc(sbase + C::OFF_V, 16, 1024);          // V, K-major (A of dP^T)
        const uint64_t dK_mn = sw128_desc(sbase + C::OFF_K, kBK * 128, 1024);  // K, d contiguous
        const uint64_t dS_k = sw128_desc(sbase + C::OFF_DS, 16, 1024);         // dS^T, K-major (A of dK)
        const uint64_t dS_mn = sw128_desc(sbase + C::OFF_DS, kBK * 128, 1024); // dS^T, q contiguous
        // S^T (A = K) or dP^T (A = V) over D from a Q / dO tile whose 64-column chunks lie
        // chunk_stride bytes apart.
        // Loops over 64-column chunks stay rolled (the descriptors advance by one add per
        // chunk) and the four 16-deep MMAs of a chunk are unrolled: compact code that still
        // issues faster than the tensor pipe retires.
        auto mma_front = [&](uint64_t a_k, uint32_t b_addr, uint32_t d_col, bool onto = false) {
          uint64_t b_k = sw128_desc(b_addr, 16, 1024);
  #pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
  #pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              mma_ss_w(tmem + d_col, desc_at(a_k, k4 * 32), desc_at(b_k, k4 * 32), idST, onto || (c | k4) != 0);
            a_k = desc_at(a_k, kBK * 128);
            b_k = desc_at(b_k, BQ * 128);
          }
        };
        // dQ of a step from dS^T in shared memory, each half of D once the drain has copied the
        // previous step's out of TMEM.
        auto mma_dq = [&](int dq_steps) -> bool {
          if constexpr (C::DQT) {
            // dQ^T[d, q] = K^T dS^T : A = K (d contiguous), B = dS^T (q contiguous)
  #pragma unroll 1
            for (int m = 0; m < D / 128; ++m) {
              if (dq_steps >= 1 && !mbar_wait_warp(dq_empty(m), (dq_steps - 1) & 1, p.status)) return false;
              tc_fence_after();
              const uint64_t a_m = desc_at(dK_mn, (2 * m) * (kBK * 128));
  #pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                mma_ss_w(tmem + C::TM_DQ + m * BQ, desc_at(a_m, kk * 2048), desc_at(dS_mn, kk * 2048), idDQ, kk > 0);
            }
          } else {
            // dQ[q, d] = dS K : A = dS (q contiguous), B = K (d contiguous)
            if (dq_steps >= 1 && !mbar_wait_warp(dq_empty(0), (dq_steps - 1) & 1, p.status)) return false;
            tc_fence_after();
  #pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_ss_w(tmem + C::TM_DQ, desc_at(dS_mn, kk * 2048), desc_at(dK_mn, kk * 2048), idDQ, kk > 0);
          }
          return true;
        };
        bool ok = mbar_wait_warp(kv_full, 0, p.status);
        int dq_steps = 0;
        if constexpr (C::TWO) {
          // dK-pass step i: Q_i in ring slot i & 1 (its use i >> 1), dO_i in slot 2 (use i), dS^T
          // in buffer i & 1.
          const uint64_t dS_k1 = sw128_desc(sbase + C::OFF_DS1, 16, 1024);
          const uint64_t dS_mn1 = sw128_desc(sbase + C::OFF_DS1, kBK * 128, 1024);
          // dV of a dV-pass step: P^T from TMEM, dO of its slot; releases that dO slot.
          auto back_dv = [&](int jj) -> bool {
            const int s = slot_of(jj);
            if (!mbar_wait_warp(do_full(s), use_of(jj) & 1, p.status)) return false;
            tc_fence_after();
            const uint64_t o_mn = sw128_desc(do_addr(s), BQ * 128, 1024);
  #pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
              mma_ts_w(tmem + C::TM_DV, tmem + C::TM_P + kk * 8, desc_at(o_mn, kk * 2048), idKV,
                       (jj > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(do_empty(s));
            mma_commit_w(mma_done);
            mma_commit_w(mma_done);  // both arrivals of the step: no dK in the dV pass
            return true;
          };
          // dK of a dK-pass step (front warp): from Q of the step, still in its ring slot (waited
          // on by the step's S^T), in two N = 128 halves of D (each a 16 KiB run of the tile);
          // releases the slot.
          auto mma_dk = [&](int jj) -> bool {
            const int i = jj - nper, r = i & 1;
            const uint64_t dsk = r ? dS_k1 : dS_k;
  #pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
              const uint64_t q_mn = sw128_desc(ring_addr(r) + hf * (C::QT_BYTES / 2), BQ * 128, 1024);
  #pragma unroll
              for (int kk = 0; kk < BQ / 16; ++kk)
                mma_ss_w(tmem + C::TM_DK + hf * (D / 2), desc_at(dsk, (kk >> 2) * (kBK * 128) + (kk & 3) * 32),
                         desc_at(q_mn, kk * 2048), idKh, (jj > nper || kk > 0) ? 1u : 0u);
            }
            mma_commit_w(ring_empty(r));
            mma_commit_w(dsb_done(r));
            return true;
          };
          // dQ^T of a dK-pass step (back warp), one 128-row half of D at a time in the same 64
          // columns, each once the drain has copied the previous half out.
          auto back_dq = [&]() -> bool {
            const int x = dq_steps & 1;  // dK-pass step dq_steps reads dS^T buffer x
            const uint64_t dsmn = x ? dS_mn1 : dS_mn;
  #pragma unroll 1
            for (int m = 0; m < 2; ++m) {
              const int hh = 2 * dq_steps + m;
              if (hh >= 1 && !mbar_wait_warp(dq_empty(0), (hh - 1) & 1, p.status)) return false;
              tc_fence_after();
              const uint64_t a_m = desc_at(dK_mn, (2 * m) * (kBK * 128));
  #pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                mma_ss_w(tmem + C::TM_DQH, desc_at(a_m, kk * 2048), desc_at(dsmn, kk * 2048), idDQ, kk > 0);
              mma_commit_w(dq_full);
            }
            ++dq_steps;
            mma_commit_w(dsb_done(x));
            return true;
          };
          // Waits for use u of ring slot r (the front warp is its only reader, in fill order).
          auto ring_wait = [&](int r, int u) -> bool {
            if (!mbar_wait_warp(ring_full(r), u & 1, p.status)) return false;
            tc_fence_after();
            return true;
          };
          if (!back_warp) {
            // Front: S^T of every step (dV pass: from its Q stage, which is free again right
            // after); in the dK pass S^T_i (once the softmax has copied dP^T_{i-1} out of the
            // shared score buffer), dK of the previous step (once its dS is in), then
            // dP^T_i = V dO_i^T with V in TMEM (once S^T_i is copied out): the softmax works on a
            // step while dK / dQ of the one before run.
            for (int j = 0; ok && j < nper; ++j) {
              if (j >= 1 && !mbar_wait_warp(sdp_free, (j - 1) & 1, p.status)) break;
              const int s = slot_of(j);
              if (!mbar_wait_warp(qdo_full(s), use_of(j) & 1, p.status)) break;
              tc_fence_after();
              mma_front(dK_k, slot_addr(s), C::TM_S);
              mma_commit_w(s_full);
              mma_commit_w(qdo_empty(s));
            }
            for (int j = nper; ok && j < nsteps; ++j) {
              const int i = j - nper;
              if (i == 0) {
                // the last dV-pass scores are read, and dV is stored (its accumulator becomes
                // dK's, P's columns become the score buffer)
                if (nper >= 1 && !mbar_wait_warp(sdp_free, (nper - 1) & 1, p.status)) break;
                if (!mbar_wait_warp(acc_free, 0, p.status)) break;
              } else if (!mbar_wait_warp(dp_free, (i - 1) & 1, p.status)) {
                break;
              }
              if (!ring_wait(i & 1, i >> 1)) break;
              mma_front(dK_k, ring_addr(i & 1), C::TM_SDP);
              mma_commit_w(s_full);
              if (i >= 1) {  // dK of the previous step as soon as its dS is in: frees its Q slot
                if (!mbar_wait_warp(p_ready_b((i - 1) & 1), ((i - 1) >> 1) & 1, p.status)) break;
                tc_fence_after();
                if (!mma_dk(j - 1)) break;
              }
              if (!mbar_wait_warp(sdp_free, j & 1, p.status)) break;
              if (i == 0 && !mbar_wait_warp(v_full, 0, p.status)) break;
              if (!ring_wait(2, i)) break;
              {  // dP^T = V dO^T: A = V from TMEM (bf16 pairs along D), B = dO (K-major chunks)
                uint64_t b_k = sw128_desc(ring_addr(2), 16, 1024);
  #pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
  #pragma unroll
                  for (int k4 = 0; k4 < 4; ++k4)
                    mma_ts_w(tmem + C::TM_SDP, tmem + C::TM_V + c * 32 + k4 * 8, desc_at(b_k, k4 * 32), idST,
                             (c | k4) != 0 ? 1u : 0u);
                  b_k = desc_at(b_k, BQ * 128);
                }
              }
              mma_commit_w(ring_empty(2));
              mma_commit_w(dp_full);
            }
            const int nB = nsteps - nper;
            if (ok && nB > 0 && mbar_wait_warp(p_ready_b((nB - 1) & 1), ((nB - 1) >> 1) & 1, p.status)) {
              tc_fence_after();
              mma_dk(nsteps - 1);
            }
          } else {
            // Back: dV (dV pass) or dQ (dK pass) of step j - 1 once its P or dS is in.
            for (int j = 1; ok && j <= nsteps; ++j) {
              const int jj = j - 1, i = jj - nper;
              if (!(jj < nper ? mbar_wait_warp(p_ready, jj & 1, p.status)
                              : mbar_wait_warp(p_ready_b(i & 1), (i >> 1) & 1, p.status)))
                break;
              tc_fence_after();
              if (!(jj < nper ? back_dv(jj) : back_dq())) break;
            }
          }
        } else {
          // dV / dK / dQ of step jj (P^T in TMEM and dS^T in shared memory are ready).
          auto issue_back = [&](int jj) -> bool {
            const int s = slot_of(jj);
            const uint64_t q_mn = sw128_desc(slot_addr(s), BQ * 128, 1024);
            const uint64_t o_mn = desc_at(q_mn, C::QT_BYTES);
  #pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)  // dV += P^T dO
              mma_ts_w(tmem + C::TM_DV, tmem + C::TM_P + kk * 8, desc_at(o_mn, kk * 2048), idKV,
                       (jj > 0 || kk > 0) ? 1u : 0u);
  #pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)  // dK += dS^T Q
              mma_ss_w(tmem + C::TM_DK, desc_at(dS_k, (kk >> 2) * (kBK * 128) + (kk & 3) * 32),
                       desc_at(q_mn, kk * 2048), idKV, (jj > 0 || kk > 0) ? 1u : 0u);
            if (!mma_dq(dq_steps)) return false;
            mma_commit_w(dq_full);
            ++dq_steps;
            mma_commit_w(mma_done);
            mma_commit_w(qdo_empty(s));
            return true;
          };
          // S^T and dP^T of step j.
          auto issue_front = [&](int j) -> bool {
            const int s = slot_of(j);
            if (!mbar_wait_warp(qdo_full(s), use_of(j) & 1, p.status)) return false;
            tc_fence_after();
            mma_front(dK_k, slot_addr(s), C::TM_S);
            // dP^T := -D (the ones tile: both offsets 128 bytes, every row reads ones), then
            // += V dO^T.
            mma_ss_w(tmem + C::TM_DP, plain_desc(sbase + C::OFF_ONES, 128, 128),
                     plain_desc(sbase + C::OFF_DSP + s * C::DSP_BYTES, BQ * 16, 128), idST, 0u);
            mma_front(dV_k, slot_addr(s) + C::QT_BYTES, C::TM_DP, true);
            mma_commit_w(s_full);
            return true;
          };
          // Front: S^T / dP^T of step j as soon as the softmax has copied step j - 1's out of
          // TMEM (sdp_free) and its stage is loaded.  Back: dV / dK / dQ of step j - 1 once its
          // P and dS are in place (p_ready); they release the stage.
          if (!back_warp) {
            for (int j = 0; ok && j < nsteps; ++j) {
              if (j >= 1) {
                if (!mbar_wait_warp(sdp_free, (j - 1) & 1, p.status)) break;
                tc_fence_after();
              }
              if (!issue_front(j)) break;
            }
          } else {
            for (int j = 1; ok && j <= nsteps; ++j) {
              if (!mbar_wait_warp(p_ready, (j - 1) & 1, p.status)) break;
              tc_fence_after();
              if (!issue_back(j - 1)) break;
            }
          }
        }
        mma_commit_w(fin_done);  // every MMA issued by this CTA has completed
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegDrain));
    // ------------------------------------------------------------ dQ drain warps
    // One thread waits on the mbarriers and the four warps follow it through a named
    // barrier, so their exits stay uniform.
    const int wq = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const int row = wq * 32 + lane;  // TMEM lane: a d index (dQ^T) or a query row (dQ)
    const int t = threadIdx.x - 384;
    int *flag = misc_i + 13;
    float *stage = reinterpret_cast<float *>(smem + C::OFF_DQS);
    const uint32_t stage_a = sbase + C::OFF_DQS;
    int dq_steps = 0;
    for (int j = 0; j < nsteps; ++j) {
      if (step_kind(j) == 1) continue;
      const int h = step_h(j), q0 = step_q0(j);
      if constexpr (C::TWO) {
        // dK pass: one 128-row half of dQ^T at a time in 64 columns; each half is released
        // once its two 32-query chunks are in registers, then leaves through [128 d, 32 q]
        // boxes staged in shared memory for bulk reduce-adds into the fp32 accumulator.
        bool okh = true;
#pragma unroll 1
        for (int m = 0; m < 2 && okh; ++m) {
          const int hh = 2 * dq_steps + m;
          if (t == 0) *flag = mbar_wait(dq_full, hh & 1, p.status) ? 1 : 0;
          named_bar<2, 128>();
          okh = *flag != 0;
          if (!okh) break;
          tc_fence_after();
          uint32_t v0[32], v1[32];
          tmem_ld32(lane_addr + C::TM_DQH, v0);
          tmem_ld32(lane_addr + C::TM_DQH + 32, v1);
          tmem_wait_ld();
          reg_fence(v0);
          reg_fence(v1);
          tc_fence_before();
          mbar_arrive(dq_empty(0));  // this thread is done with the half
          // four [128 d, 16 q] boxes through four 8 KiB buffers, so that staging a box
          // overlaps the reduce-adds of the ones before
#pragma unroll
          for (int bx = 0; bx < 4; ++bx) {
            const int boff = bx < 2 ? C::OFF_DQS + bx * 8192 : C::OFF_DQS2 + (bx - 2) * 8192;
            float *sb = reinterpret_cast<float *>(smem + boff);
            if (t == 0) bulk_wait_read_but<3>();  // the box four back has left this buffer
            named_bar<2, 128>();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              sb[e * 128 + row] = __uint_as_float(bx < 2 ? v0[(bx & 1) * 16 + e] : v1[(bx & 1) * 16 + e]);
            fence_async_smem();
            named_bar<2, 128>();
            if (t == 0) {
              tma_reduce_add_4d(&tmDQ, sbase + boff, m * 128, q0 + bx * 16, h, b);
              bulk_commit();
            }
          }
        }
        if (!okh) break;
        ++dq_steps;
        continue;
      }
      if (t == 0) *flag = mbar_wait(dq_full, dq_steps & 1, p.status) ? 1 : 0;
      named_bar<2, 128>();
      if (!*flag) break;
      tc_fence_after();
      if constexpr (C::DQT) {
        // dQ^T: lane = d within a 128-wide half of D, column = query.  32 queries at a time go
        // to registers (a half of D is released once its last 32 are in: the next step's dQ
        // MMAs for that half may start), then leave through a [128 d, 32 q] box staged in
        // shared memory for a bulk reduce-add into the fp32 accumulator.
#pragma unroll 1
        for (int c = 0; c < C::DQ_COLS / 32; ++c) {
          const int m = c / (BQ / 32), cq = c % (BQ / 32);
          uint32_t v[32];
          tmem_ld32(lane_addr + C::TM_DQ + c * 32, v);
          tmem_wait_ld();
          reg_fence(v);
          if (cq == BQ / 32 - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty(m));  // this thread is done with this half of the TMEM tile
          }
          if (t == 0) bulk_wait_read_all();  // the previous box has left shared memory
          named_bar<2, 128>();
#pragma unroll
          for (int e = 0; e < 32; ++e) stage[e * 128 + row] = __uint_as_float(v[e]);
          fence_async_smem();
          named_bar<2, 128>();
          if (t == 0) {
            tma_reduce_add_4d(&tmDQ, stage_a, m * 128, q0 + cq * 32, h, b);
            bulk_commit();
          }
        }
      } else {
        // dQ: lane = query row, column = d.  32 columns of d at a time (the tile is released
        // once the last of them is in), staged as [32 d, 128 q] boxes (128-byte swizzled) for
        // bulk reduce-adds.
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_addr + C::TM_DQ + c * 32, v);
          tmem_wait_ld();
          reg_fence(v);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty(0));  // this thread is done with the TMEM tile
          }
          if (t == 0) bulk_wait_read_all();
          named_bar<2, 128>();
          uint8_t *rowp = reinterpret_cast<uint8_t *>(stage) + row * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4 *>(rowp + ((u ^ (row & 7)) << 4)) =
                make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          fence_async_smem();
          named_bar<2, 128>();
          if (t == 0) {
            tma_reduce_add_4d(&tmDQ, stage_a, c * 32, q0, h, b);
            bulk_commit();
          }
        }
      }
      ++dq_steps;
    }
    if (t == 0) bulk_wait_all();
  }

  __syncwarp();  // every warp reconverges (producer and drain lanes finish at different times)
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <class C>
cudaError_t launch_bwd(const Params &p, cudaStream_t st) {
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_tmap_bshd(&tq, p.q, C::D, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb, C::BQ) ||
      !make_tmap_bshd(&tk, p.k, C::D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, kBK) ||
      !make_tmap_bshd(&tv, p.v, C::D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb, kBK) ||
      !make_tmap_bshd(&tdo, p.dO, C::D, p.Sq, p.Hq, p.B, (long long)p.Hq * C::D, C::D,
                      (long long)p.Sq * p.Hq * C::D, C::BQ) ||
      !make_tmap_f32_bshd(&tdq, p.dQacc, C::D, p.Sq, p.Hq, p.B, C::DQT ? 128 : 32, C::DQT ? (C::TWO ? 16 : 32) : 128,
                          !C::DQT))
    return cudaErrorInvalidValue;
  // The group-major order is built for the two-pass form (head dim 256), where it was measured.
  const bool gm = C::TWO && p.bwd_group_major;
  auto kern = p.bias ? (p.cap > 0.f ? bwd_tc_kernel<C, true, true, false> : bwd_tc_kernel<C, false, true, false>)
                     : (p.cap > 0.f ? bwd_tc_kernel<C, true, false, false> : bwd_tc_kernel<C, false, false, false>);
  if constexpr (C::TWO) {
    if (gm)
      kern = p.bias ? (p.cap > 0.f ? bwd_tc_kernel<C, true, true, true> : bwd_tc_kernel<C, false, true, true>)
                    : (p.cap > 0.f ? bwd_tc_kernel<C, true, false, true> : bwd_tc_kernel<C, false, false, true>);
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const long long nblk = (long long)((p.Sk + kBK - 1) / kBK) * p.Hkv * p.B;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidValue;
  Params q = p;
  if (!follow_work_list(nblk)) q.korder = nullptr;
  kern<<<(unsigned)nblk, kThreads, C::SMEM, st>>>(tq, tk, tv, tdo, tdq, q);
  return counted(cudaGetLastError());
}

}  // namespace

bool tc_bwd_supported(int D) { return D == 64 || D == 128 || D == 256; }
bool tc_bwd_fused(int D) { return D == 64 || D == 128; }

cudaError_t tc_backward(const Params &p, cudaStream_t st) {
  switch (p.D) {
    case 64: return launch_bwd<BwdCfg<64, 128, false, false, 3>>(p, st);
    case 128: return launch_bwd<BwdCfg<128, 64, true, false, 3>>(p, st);
    case 256: return launch_bwd<BwdCfg<256, 64, true, true, 1>>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
