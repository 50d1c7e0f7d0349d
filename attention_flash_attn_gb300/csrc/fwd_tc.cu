// fwd_tc.cu -- tcgen05 tensor-core forward for bf16, D in {64, 128, 256} and the wide form (320 .. 512).
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   warp 0      TMA producers: the Q tile once, then K tiles (lane 0) and V tiles (lane 1)
//               into separate rings, each slot released as soon as its MMA has read it;
//   warp 1      MMA issuer (one elected lane of the converged warp) and TMEM owner: S_j = Q K_j^T into one of two TMEM
//               score buffers, then O += P_{j-1} V_{j-1} with P read from TMEM;
//   warps 2..9  softmax: a query row is a TMEM lane, and the two warps that share a lane
//               quarter split its BN key columns.  Per KV tile each thread reads its half
//               row of S, applies scale, the tanh soft-cap and the mask, exchanges its half
//               row maximum with its partner through shared memory, keeps a running max /
//               sum (started from the sink column, so the sink enters the row exactly once),
//               writes P as bf16 over the score buffer, and rescales its half of the O
//               accumulator in TMEM only when the running max grew by more than 2^8.  At the
//               end the two halves' sums are combined, O is normalised and stored (bf16) with
//               LSE (natural log).
// The score modification follows the soft-capping pages: cap * tanh(u / cap) applied after
// the scale and before the mask (TransformerEngine PR #3391; tokamax PR #1121).  The sink
// column's role follows TransformerEngine PR #3551 ("What changed").
//
// Every mbarrier wait is bounded: a wait that gives up records kStatusWaitTimeout in the
// status word and the CTA winds down without trapping.  The partner exchange carries each
// thread's failure flag, so both warps of a pair leave together.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // tolerate P <= 2^8 before rescaling O

// Wide form (NV == 0; head dims 320, 384, 448 and 512, instantiated once with D = 512 as the
// capacity and the head dim read at run time): S = Q K^T needs all of D, but O would take every
// TMEM column, so each CTA produces one part of O -- the head-dim chunking above 256 of the
// MaxText commit message quoted on tokamax PR #1121: of the D / 64 column chunks, the first
// CTA of a pair takes the first ceil(D / 128), the second the rest -- and S is computed by both
// CTAs.  Q stays resident (up to 128 KiB); K and V tiles stream through one ring of NK 32 KiB
// slots, each slot two 64-column chunks of a 128-key tile (the last slot of an odd chunk count
// holds one), loaded and consumed in the MMA warp's order.
template <int D, int BN, int NK, int NV>
struct FwdCfg {
  static constexpr bool WIDE = NV == 0;
  static constexpr int DV = WIDE ? D / 2 : D;           // O columns this CTA produces (wide: at most)
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int KV_BYTES = WIDE ? 2 * BN * 128 : BN * D * 2;  // wide: one ring slot
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;                 // NK-deep K ring (released after S)
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;   // NV-deep V ring (released after PV)
  static constexpr int OFF_X = OFF_V + NV * KV_BYTES;   // partner exchange: [2 halves][3 slots][128] floats
  static constexpr int OFF_BAR = OFF_X + 6 * kBM * 4;
  // One K and one V tile (head dim 256): each is moved and released in two halves with
  // barriers of their own -- K by head-dim halves (chunks 0-1, 2-3), V by key halves (rows
  // 0-63, 64-127, the halves the PV MMAs read in turn) -- so that a step's MMAs start on the
  // first half while the second lands, and the next tile's first half loads while the second
  // is still read.
  static constexpr bool HALF = NK == 1 && NV == 1;
  static constexpr int RK = HALF ? 2 : NK, RV = HALF ? 2 : NV;  // barrier pairs per ring
  static constexpr int NBAR = 1 + 2 * RK + 2 * RV + 6;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static constexpr int TM_O = 2 * BN;
  // Tensor memory: two score buffers and O; when they fit 256 columns and shared memory leaves
  // room, two CTAs share an SM (MINB), so that one's softmax overlaps the other's MMAs.
  static constexpr int TM_COLS = 2 * BN + DV <= 256 ? 256 : 512;
  static constexpr int MINB = (TM_COLS == 256 && OFF_MISC + 64 + 1024 <= 113 * 1024) ? 2 : 1;
  static constexpr int HC = BN / 2;  // columns per softmax thread and tile
  static_assert(2 * BN + DV <= TM_COLS, "TMEM budget");
  static_assert(!WIDE || (BN == 128 && D % 128 == 0 && DV % 128 == 0), "wide form: 128-key tiles, 128-column slots");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(KV_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzle atoms must stay 1 KiB aligned");
  static_assert(HC % 32 == 0, "half rows are whole 32-column TMEM loads");
};

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int e = 0; e < N; ++e) asm volatile("" : "+r"(r[e]));
}

// TMEM column (relative to its score buffer) of the bf16 P pairs that the PV MMA's 16-key
// slice kk reads: the softmax half owning keys 16 kk .. 16 kk + 15 (HC keys per half) wrote
// its P over the first HC / 2 columns of its own HC score columns.
template <int HC>
__device__ __forceinline__ constexpr uint32_t p_col(int kk) {
  return (uint32_t)(kk * 8 + (kk * 16 / HC) * (HC / 2));
}

// Pair barrier of the two softmax warps that share TMEM lane quarter `wq` (ids 2..5).  The
// aligned form needs each warp converged when it arrives: the __syncwarp makes it so, whatever
// per-lane waits or branches came before.
__device__ __forceinline__ void pair_bar(int wq) {
  __syncwarp();
  asm volatile("bar.sync %0, 64;" ::"r"(2 + wq) : "memory");
}

// Score constants as packed pairs.  With the soft-cap, e = exp(2 u / cap) for u = scale s and
// r = 1 / (1 + e): tanh(u / cap) = 1 - 2 r, so the capped logit in log2 units is
// cap log2(e) (1 - 2 r), with r from f2_sigmoid2_neg (FMA-pipe reciprocal).  A huge e (its
// exponent is clamped at 126) gives r ~ 0 (tanh = 1), an underflowing one r = 1.
// With a bias the logit is u = scale s + bias; the bias enters as its own term (bin: its
// factor, 2 log2(e) / cap with the cap, log2(e) without).  `off` (the fixed exponent offset,
// else 0) is subtracted from the capped logit in the same FMA.
struct FwdScore {
  uint64_t cin, mcap2, cap2, sc2, bin;
  __device__ FwdScore(float scale, float inv_cap, float cap, float off) {
    cin = f2_splat(2.f * kLog2e * scale * inv_cap);
    mcap2 = f2_splat(-2.f * cap * kLog2e);
    cap2 = f2_splat(cap * kLog2e - off);
    sc2 = f2_splat(scale * kLog2e);
    bin = f2_splat(cap > 0.f ? 2.f * kLog2e * inv_cap : kLog2e);
  }
};

// The bias of one bf16 pair (low half first) as a pair of floats.
__device__ __forceinline__ uint64_t bias_pair(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// This thread's N2 bias pairs of a tile: row `row`, columns j0 .. j0 + 2 N2 - 1; columns at
// or past Sk read as 0 (they are masked).  16-byte loads when every row starts on a 16-byte
// boundary and the columns lie inside the row.  The branch depends on warp-uniform values only,
// so the warp stays converged for the tensor-memory instructions that follow.
template <int N2>
__device__ __forceinline__ void load_bias_row(uint32_t (&bq)[N2], const __nv_bfloat16 *row, int j0, int Sk,
                                              bool vec) {
  if (vec && j0 + 2 * N2 <= Sk) {
    const uint4 *src = reinterpret_cast<const uint4 *>(row + j0);
#pragma unroll
    for (int v = 0; v < N2 / 4; ++v) {
      const uint4 x = __ldg(src + v);
      bq[4 * v] = x.x;
      bq[4 * v + 1] = x.y;
      bq[4 * v + 2] = x.z;
      bq[4 * v + 3] = x.w;
    }
  } else {
    const unsigned short *r16 = reinterpret_cast<const unsigned short *>(row);
#pragma unroll
    for (int e = 0; e < N2; ++e) {
      const int ja = j0 + 2 * e;  // clamped indices: every load stays inside the row
      const uint32_t lo = __ldg(r16 + min(ja, Sk - 1)), hi = __ldg(r16 + min(ja + 1, Sk - 1));
      bq[e] = (ja < Sk ? lo : 0u) | (ja + 1 < Sk ? hi << 16 : 0u);
    }
  }
}

// Raw scores -> capped, masked base-2 logits (less the score's offset) in place; returns their
// maximum.  MIX: every other pair takes the cap's reciprocal from the special-function unit
// (rcp.approx) instead of the FMA pipe -- 5 issue slots per pair instead of 11, for two more
// special-function ops -- for kernels whose softmax warps are issue-bound with that unit part
// idle.  That form needs no clamp: an exponential that overflows to +inf gives 1 / inf = 0,
// the cap's own limit (the FMA-pipe reciprocal's bit-level seed needs a finite input).
template <bool CAP, bool MASKED, bool MIX, bool BIAS, int N>
__device__ __forceinline__ float logits2(uint32_t (&x)[N], const FwdScore &k, int jbase, int lo, int hi,
                                         bool pairwise, const int *segk, int sid, const uint32_t *bq) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    const uint64_t s2 = f2_pack(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
    uint64_t t2;
    if constexpr (CAP) {
      const uint64_t x2 = BIAS ? f2_fma(s2, k.cin, f2_mul(bias_pair(bq[e / 2]), k.bin)) : f2_mul(s2, k.cin);
      uint64_t r2;
      if (MIX && (e & 2)) {
        float xa, xb, da, db;
        f2_unpack(x2, xa, xb);
        f2_unpack(f2_add(f2_pack(ex2_approx(xa), ex2_approx(xb)), f2_splat(1.f)), da, db);
        r2 = f2_pack(rcp_approx(da), rcp_approx(db));
      } else {
        r2 = f2_sigmoid2_neg(x2);
      }
      t2 = f2_fma(r2, k.mcap2, k.cap2);
    } else {
      t2 = BIAS ? f2_fma(s2, k.sc2, f2_mul(bias_pair(bq[e / 2]), k.bin)) : f2_mul(s2, k.sc2);
    }
    float ta, tb;
    f2_unpack(t2, ta, tb);
    if constexpr (MASKED) {
      const int ja = jbase + e, jb = ja + 1;
      bool va = ja >= lo && ja < hi, vb = jb >= lo && jb < hi;
      if (pairwise) {
        va = va && __ldg(segk + ja) == sid;
        vb = vb && __ldg(segk + jb) == sid;
      }
      ta = va ? ta : -INFINITY;
      tb = vb ? tb : -INFINITY;
    }
    x[e] = __float_as_uint(ta);
    x[e + 1] = __float_as_uint(tb);
    m0 = fmaxf(m0, ta);
    m1 = fmaxf(m1, tb);
  }
  return fmaxf(m0, m1);
}

// FIXM (soft-cap on, cap <= kFixedMaxCap): every capped logit lies in [-cap, cap], so the row's
// exponent offset is fixed up front instead of tracked -- no running maximum, no partner
// exchange of maxima, no rescaling of O.  Softmax is invariant to the offset.  In log2 units the
// offset is max(cap - delta, sink) with delta = max(0, 2 cap - 124): the smallest visible
// probability (2^(delta - 2 cap) without a sink) stays a normal float, and the largest is at
// most 2^delta <= 2^32 (the tracked form lets P reach 2^8 before it rescales).  With a larger
// sink the sink's own term (1) dominates the row sum, so probabilities that underflow there are
// negligible.
constexpr float kFixedMaxCap = 54.0f;  // 2 cap log2(e) - 124 <= 32
__device__ __forceinline__ float fixed_delta(float cap) { return fmaxf(0.f, 2.f * cap * kLog2e - 124.f); }

template <int D, int BN, int NK, int NV, bool CAP, bool FIXM, bool BIAS>
__global__ void __launch_bounds__(kThreads, FwdCfg<D, BN, NK, NV>::MINB)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = FwdCfg<D, BN, NK, NV>;
  constexpr int HC = C::HC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *misc_i = reinterpret_cast<int *>(smem + C::OFF_MISC);
  {  // A wait elsewhere already gave up: do nothing (decided once for the whole CTA; the
     // caller learns it from the status word).
    if (threadIdx.x == 0) misc_i[12] = (status_peek(p.status) & kStatusWaitTimeout) ? 1 : 0;
    __syncthreads();
    if (misc_i[12]) return;
  }

  // One-dimensional grid, heaviest tiles first so that the last wave holds the light ones.
  // With segments the order is the mask metadata's longest-first work list of (batch, query
  // tile) pairs, every head of a pair adjacent; otherwise the query tile varies slowest,
  // latest (heaviest under causal masks, equal under a window alone) first.  With a split-KV
  // forward the split index varies fastest.
  const int nqt = (p.Sq + kBM - 1) / kBM;
  const int ns = p.kv_splits > 1 ? p.kv_splits : 1;
  // Wide form: the two CTAs of a (query tile, head) pair -- one per half of O -- are adjacent.
  constexpr int NVH = C::WIDE ? 2 : 1;
  const int vh = (int)(blockIdx.x % (unsigned)NVH);
  const unsigned bx = blockIdx.x / (unsigned)NVH;
  int qt, b, h, split;
  if (p.qorder) {
    const int2 o = p.qorder[bx / (unsigned)(p.Hq * ns)];
    const int hs = (int)(bx % (unsigned)(p.Hq * ns));
    b = o.x;
    qt = o.y;
    h = hs / ns;
    split = hs % ns;
  } else {
    const int bhs = (int)(bx % (unsigned)(p.Hq * p.B * ns));
    qt = nqt - 1 - (int)(bx / (unsigned)(p.Hq * p.B * ns));
    split = bhs % ns;
    const int bh = bhs / ns;
    h = bh % p.Hq;
    b = bh / p.Hq;
  }
  const int g = h / p.G;
  const int i0 = qt * kBM, i1 = min(i0 + kBM, p.Sq) - 1;
  const int off = p.Sk - p.Sq;
  // 64-column chunks of D that S runs over, and this CTA's chunks of O: vcn of them from vc0.
  const int nch = C::WIDE ? p.D / 64 : C::KCH;
  const int vc0 = (C::WIDE && vh == 1) ? (nch + 1) / 2 : 0;
  const int vcn = C::WIDE ? (vh == 0 ? (nch + 1) / 2 : nch / 2) : C::DV / 64;

  // Keys this query tile can see (uniform across the CTA).
  int klo = 0, khi = p.Sk;
  if (!p.qoff) {  // per-sequence offsets: the tile ranges below carry the causal / window bounds
    if (p.window > 0) klo = max(klo, i0 + off - p.window + 1);
    if (p.causal) khi = min(khi, i1 + off + 1);
  }
  if (p.qtile) {  // the tile's class bounds from the mask metadata
    const int4 c = p.qtile[(size_t)b * nqt + qt];
    klo = max(klo, c.x);
    khi = min(khi, c.y);
  }
  const int tv0 = klo / BN;
  const int nv = (klo < khi) ? (khi + BN - 1) / BN - tv0 : 0;
  // Split s of ns takes key tiles [tv0 + s nv / ns, tv0 + (s + 1) nv / ns) of the visible ones.
  const int t0 = tv0 + (int)((long long)split * nv / ns);
  const int n = tv0 + (int)((long long)(split + 1) * nv / ns) - t0;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0;
  constexpr int RK = C::RK, RV = C::RV;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + RK + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * RK + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * RK + RV + s); };
  auto s_full = [&](int x) { return bar0 + 8u * (1 + 2 * RK + 2 * RV + x); };
  auto p_full = [&](int x) { return bar0 + 8u * (3 + 2 * RK + 2 * RV + x); };
  const uint32_t o_done = bar0 + 8u * (5 + 2 * RK + 2 * RV);
  const uint32_t o_fin = bar0 + 8u * (6 + 2 * RK + 2 * RV);  // FIXM: every PV MMA has completed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *red = misc_i + 4;  // [8]
  float *xbuf = reinterpret_cast<float *>(smem + C::OFF_X);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < RK; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < RV; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), kSoftmaxThreads);
    }
    mbar_init(o_done, 1);
    mbar_init(o_fin, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0 && (tmem & 0xFFFFu) + C::TM_COLS > 512) set_status(p.status, kStatusBadTmemAlloc);

  if (warp == 0 && C::WIDE) {
    // ------------------------------------------------------------ TMA producer (wide form)
    // Lane 0 loads Q, then every K and V slot in the order the MMA warp reads them: K_j for
    // S_j, then V_{j-1} (this CTA's half of O) for PV_{j-1}.
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, nch * (kBM * 128));
#pragma unroll 1
      for (int c = 0; c < nch; ++c)
        tma_load_4d(sbase + C::OFF_Q + c * (kBM * 128), &tmQ, q_full, c * 64, i0, h, b);
      int u = 0;  // ring uses so far
      // One slot: chunk c of `tm` (columns 64 c ..), and chunk c + 1 when `two`.
      auto slot_load = [&](const CUtensorMap *tm, int c, int row, bool two) -> bool {
        const int s = u % NK;
        if (u >= NK && !mbar_wait(k_empty(s), ((u / NK) - 1) & 1, p.status)) return false;
        mbar_arrive_expect_tx(k_full(s), two ? C::KV_BYTES : C::KV_BYTES / 2);
        tma_load_4d(sbase + C::OFF_K + s * C::KV_BYTES, tm, k_full(s), c * 64, row, g, b);
        if (two) tma_load_4d(sbase + C::OFF_K + s * C::KV_BYTES + BN * 128, tm, k_full(s), c * 64 + 64, row, g, b);
        ++u;
        return true;
      };
      bool okp = true;
      for (int j = 0; okp && j <= n; ++j) {
        if (j < n)
          for (int c = 0; okp && c < nch; c += 2) okp = slot_load(&tmK, c, (t0 + j) * BN, c + 1 < nch);
        if (j >= 1)
          for (int c = 0; okp && c < vcn; c += 2) okp = slot_load(&tmV, vc0 + c, (t0 + j - 1) * BN, c + 1 < vcn);
      }
    }
  } else if (warp == 0) {
    if constexpr (!C::WIDE) {
    // ------------------------------------------------------------ TMA producers
    // Lane 0 loads Q and the K ring, lane 1 the V ring: K slots free up as soon as their S
    // MMA is done, V slots only after PV, so the two rings advance independently.
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d(sbase + C::OFF_Q + c * (kBM * 128), &tmQ, q_full, c * 64, i0, h, b);
      for (int j = 0; j < n; ++j) {
        const int kt = (t0 + j) * BN;
        if constexpr (C::HALF) {
          bool okh = true;
          for (int hf = 0; hf < 2 && okh; ++hf) {  // head-dim chunks 2 hf, 2 hf + 1
            if (j >= 1 && !mbar_wait(k_empty(hf), (j - 1) & 1, p.status)) { okh = false; break; }
            mbar_arrive_expect_tx(k_full(hf), C::KV_BYTES / 2);
#pragma unroll
            for (int c = 2 * hf; c < 2 * hf + 2; ++c)
              tma_load_4d(sbase + C::OFF_K + c * (BN * 128), &tmK, k_full(hf), c * 64, kt, g, b);
          }
          if (!okh) break;
        } else {
          const int s = j % NK;
          if (j >= NK && !mbar_wait(k_empty(s), ((j / NK) - 1) & 1, p.status)) break;
          mbar_arrive_expect_tx(k_full(s), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(sbase + C::OFF_K + s * C::KV_BYTES + c * (BN * 128), &tmK, k_full(s), c * 64, kt, g, b);
        }
      }
    } else if (lane == 1 && n > 0) {
      tma_prefetch_desc(&tmV);
      for (int j = 0; j < n; ++j) {
        const int kt = (t0 + j) * BN;
        if constexpr (C::HALF) {
          bool okh = true;
          for (int hf = 0; hf < 2 && okh; ++hf) {  // key rows 64 hf .. 64 hf + 63 (64-row boxes)
            if (j >= 1 && !mbar_wait(v_empty(hf), (j - 1) & 1, p.status)) { okh = false; break; }
            mbar_arrive_expect_tx(v_full(hf), C::KV_BYTES / 2);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(sbase + C::OFF_V + c * (BN * 128) + hf * (64 * 128), &tmV, v_full(hf), c * 64, kt + 64 * hf,
                          g, b);
          }
          if (!okh) break;
        } else {
          const int s = j % NV;
          if (j >= NV && !mbar_wait(v_empty(s), ((j / NV) - 1) & 1, p.status)) break;
          mbar_arrive_expect_tx(v_full(s), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(sbase + C::OFF_V + s * C::KV_BYTES + c * (BN * 128), &tmV, v_full(s), c * 64, kt, g, b);
        }
      }
    }
    }
  } else if (warp == 1 && C::WIDE) {
    // ------------------------------------------------------------ MMA issuer (wide form)
    // S_j from the K slots of tile j (8 k-steps of 16 each over a slot's 128 columns of D, 4
    // over a one-chunk slot), then PV_{j-1}: one N = 128 (one-chunk slot: N = 64) MMA group per
    // V slot into its columns of O.
    if (n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, BN, false, false);
      constexpr uint32_t idO = idesc_bf16(kBM, 128, false, true);
      constexpr uint32_t idO64 = idesc_bf16(kBM, 64, false, true);
      const uint64_t dq0 = sw128_desc(sbase + C::OFF_Q, 16, 1024);
      int u = 0;
      bool ok = mbar_wait_warp(q_full, 0, p.status);
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n) {
          const uint32_t dS = tmem + (uint32_t)((j & 1) * BN);
#pragma unroll 1
          for (int c2 = 0; 2 * c2 < nch; ++c2, ++u) {
            const int s = u % NK;
            if (!mbar_wait_warp(k_full(s), (u / NK) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t qd = desc_at(dq0, (2 * c2) * (kBM * 128));
            const uint64_t kd = sw128_desc(sbase + C::OFF_K + s * C::KV_BYTES, 16, 1024);
            const int nk8 = 2 * c2 + 1 < nch ? 8 : 4;
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8)
              if (k8 < nk8)
                mma_ss_w(dS, desc_at(qd, (k8 >> 2) * (kBM * 128) + (k8 & 3) * 32),
                         desc_at(kd, (k8 >> 2) * (BN * 128) + (k8 & 3) * 32), idS, (c2 | k8) != 0);
            mma_commit_w(k_empty(s));
          }
          if (!ok) break;
          mma_commit_w(s_full(j & 1));
        }
        if (j >= 1) {
          const int jj = j - 1;
          if (!mbar_wait_warp(p_full(jj & 1), (jj >> 1) & 1, p.status)) break;
          const uint32_t pa = tmem + (uint32_t)((jj & 1) * BN);
#pragma unroll 1
          for (int c2 = 0; 2 * c2 < vcn; ++c2, ++u) {
            const int s = u % NK;
            if (!mbar_wait_warp(k_full(s), (u / NK) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dv = sw128_desc(sbase + C::OFF_K + s * C::KV_BYTES, BN * 128, 1024);
            const uint32_t id = 2 * c2 + 1 < vcn ? idO : idO64;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts_w(tmem + C::TM_O + c2 * 128, pa + p_col<HC>(kk), desc_at(dv, kk * (16 * 128)), id,
                       (jj > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(k_empty(s));
          }
          if (!ok) break;
          mma_commit_w(o_done);
        }
      }
      if (FIXM) mma_commit_w(o_fin);
    }
  } else if (warp == 1) {
    if constexpr (!C::WIDE) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; one elected lane issues each
    // MMA and commit.  Descriptors are built once and advanced by constant offsets.
    if (n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, BN, false, false);
      constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
      const uint64_t dq0 = sw128_desc(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dk0 = sw128_desc(sbase + C::OFF_K, 16, 1024);
      const uint64_t dv0 = sw128_desc(sbase + C::OFF_V, BN * 128, 1024);
      bool ok = mbar_wait_warp(q_full, 0, p.status);
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n && C::HALF) {
          const uint32_t dS = tmem + (uint32_t)((j & 1) * BN);
          uint64_t qd = dq0, kd = dk0;
          bool okh = true;
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait_warp(k_full(hf), j & 1, p.status)) { okh = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) mma_ss_w(dS, desc_at(qd, k4 * 32), desc_at(kd, k4 * 32), idS, (c | k4) != 0);
              qd = desc_at(qd, kBM * 128);
              kd = desc_at(kd, BN * 128);
            }
            mma_commit_w(k_empty(hf));
          }
          if (!okh) break;
          mma_commit_w(s_full(j & 1));
        } else if (j < n) {
          const int s = j % NK;
          if (!mbar_wait_warp(k_full(s), (j / NK) & 1, p.status)) break;
          tc_fence_after();
          const uint32_t dS = tmem + (uint32_t)((j & 1) * BN);
          // 64-column chunks rolled (one descriptor add each), their four MMAs unrolled.
          uint64_t qd = dq0, kd = desc_at(dk0, s * C::KV_BYTES);
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) mma_ss_w(dS, desc_at(qd, k4 * 32), desc_at(kd, k4 * 32), idS, (c | k4) != 0);
            qd = desc_at(qd, kBM * 128);
            kd = desc_at(kd, BN * 128);
          }
          mma_commit_w(s_full(j & 1));
          mma_commit_w(k_empty(s));
        }
        if (j >= 1 && C::HALF) {
          const int jj = j - 1;
          if (!mbar_wait_warp(p_full(jj & 1), (jj >> 1) & 1, p.status)) break;
          const uint32_t pa = tmem + (uint32_t)((jj & 1) * BN);
          bool okh = true;
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait_warp(v_full(hf), jj & 1, p.status)) { okh = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 4 * hf; kk < 4 * hf + 4; ++kk)
              mma_ts_w(tmem + C::TM_O, pa + p_col<HC>(kk), desc_at(dv0, kk * (16 * 128)), idO,
                       (jj > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(v_empty(hf));
          }
          if (!okh) break;
          mma_commit_w(o_done);
        } else if (j >= 1) {
          const int jj = j - 1, s = jj % NV;
          if (!mbar_wait_warp(v_full(s), (jj / NV) & 1, p.status)) break;
          if (!mbar_wait_warp(p_full(jj & 1), (jj >> 1) & 1, p.status)) break;
          tc_fence_after();
          const uint64_t dvs = desc_at(dv0, s * C::KV_BYTES);
          const uint32_t pa = tmem + (uint32_t)((jj & 1) * BN);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts_w(tmem + C::TM_O, pa + p_col<HC>(kk), desc_at(dvs, kk * (16 * 128)), idO,
                     (jj > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(v_empty(s));
          mma_commit_w(o_done);
        }
      }
      if (FIXM) mma_commit_w(o_fin);  // the softmax warps skip the per-step o_done phases
    }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp & 3;            // TMEM lane quarter of this warp
    const int half = (warp - 2) >> 2;   // which half of the key columns it owns
    const int r = wq * 32 + lane;
    const int i = i0 + r;
    const bool row_ok = i < p.Sq;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);

    const int ip = row_ok ? qpos(p, i) : i + off;
    int lo = 0, hi = p.Sk;
    if (p.window > 0) lo = max(lo, ip - p.window + 1);
    if (p.causal) hi = min(hi, ip + 1);
    bool seg_pairwise = false;
    int sid = 0;
    const int *segk = nullptr;
    if (p.seg_q && row_ok) {
      if (p.seg_mono[b]) {  // sorted ids: the metadata's interval for this row (its segment's run)
        const int2 x = __ldg(p.qrun + (size_t)b * p.Sq + i);
        lo = max(lo, x.x);
        hi = min(hi, x.y);
      } else {
        sid = __ldg(p.seg_q + (size_t)b * p.Sq + i);
        segk = p.seg_k + (size_t)b * p.Sk;
        seg_pairwise = true;
      }
    }
    if (!row_ok) {  // never stored; neutral for the tile classification
      lo = 0;
      hi = p.Sk;
    }
    // Keys every row of the tile sees, [cta_lo, cta_hi): key tiles inside need no mask.  The
    // mask metadata carries them (the tile class); otherwise the rows' intervals are
    // intersected here.
    int cta_lo, cta_hi;
    if (p.qtile) {
      const int4 c = p.qtile[(size_t)b * nqt + qt];
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
      asm volatile("barrier.sync 1, 256;" ::: "memory");
      cta_lo = max(max(red[0], red[1]), max(red[2], red[3]));
      cta_hi = min(min(red[4], red[5]), min(red[6], red[7]));
    }
    const bool any_pairwise = p.seg_q != nullptr && !p.seg_mono[b];

    // This row's bias (logically [B, Hq, Sq, Sk]; broadcast dimensions have stride 0).  A row
    // past Sq reads row Sq - 1 (never stored), so that every lane takes the same path.
    const __nv_bfloat16 *brow =
        BIAS ? static_cast<const __nv_bfloat16 *>(p.bias) + (size_t)b * p.bias_sb + (size_t)h * p.bias_sh +
                   (size_t)min(i, p.Sq - 1) * p.Sk
             : nullptr;
    const bool sink_col = has_sink_col(p) && ns == 1;  // split partials leave it to the merge
    float m_ref = sink_col ? sink_logit(p, h) * kLog2e : -INFINITY;  // running max (log2 units)
    float l = (sink_col && half == 0) ? 1.f : 0.f;                   // this half's sum relative to m_ref
    if (FIXM) {  // fixed offset: the cap bounds every logit
      const float m_fix = fmaxf(p.cap * kLog2e - fixed_delta(p.cap), m_ref);
      l = (sink_col && half == 0) ? ex2_approx(m_ref - m_fix) : 0.f;
      m_ref = m_fix;
    }
    // With the fixed offset the logits come out of logits2 already less it.
    const FwdScore ks(p.scale, p.inv_cap, p.cap, FIXM ? m_ref : 0.f);
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      const int j0 = (t0 + j) * BN + half * HC;
      uint32_t bq[BIAS ? HC / 2 : 1];
      if constexpr (BIAS) load_bias_row(bq, brow, j0, p.Sk, p.bias_vec != 0);  // in flight during the wait
      // Warp-uniform, so that a failed wait takes the whole warp (and, through the exchange
      // below, its partner) out of the loop together.
      const bool got = __all_sync(0xffffffffu, mbar_wait(s_full(j & 1), (j >> 1) & 1, p.status));
      tc_fence_after();
      const uint32_t sa = lane_addr + (uint32_t)((j & 1) * BN + half * HC);
      uint32_t xr[HC];
      if (got) {
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld32(sa + c * 32, *reinterpret_cast<uint32_t(*)[32]>(xr + c * 32));
        tmem_wait_ld();
        reg_fence(xr);
      }
      const bool full = !any_pairwise && (t0 + j) * BN >= cta_lo && (t0 + j + 1) * BN <= cta_hi;
      float mx = -INFINITY;
      if (got) {
        mx = full ? logits2<CAP, false, (D <= 128), BIAS>(xr, ks, j0, lo, hi, seg_pairwise, segk, sid, bq)
                  : logits2<CAP, true, (D <= 128), BIAS>(xr, ks, j0, lo, hi, seg_pairwise, segk, sid, bq);
      }
      float alpha_o = 1.f;
      bool resc = false;
      if (FIXM) {
        (void)mx;
        if (!(got && ok)) {  // the MMA warp then times out too; the CTA winds down
          ok = false;
          break;
        }
      } else {
      // Exchange half-row maxima (and failure flags, as NaN) with the partner warp; slot
      // j & 1 is rewritten two tiles later, after the partner has passed the next barrier.
      xbuf[(half * 3 + (j & 1)) * kBM + r] = (got && ok) ? mx : __int_as_float(0x7fffffff);
      pair_bar(wq);
      const float other = xbuf[((1 - half) * 3 + (j & 1)) * kBM + r];
      if (!(got && ok) || isnan(other)) {
        ok = false;
        break;
      }
      const float m_new = fmaxf(m_ref, fmaxf(mx, other));
      if (m_new != -INFINITY) {
        if (j == 0 || m_ref == -INFINITY) {
          // first finite max: O is either about to be overwritten (j == 0) or all-zero
          l = (m_ref == -INFINITY) ? 0.f : l * ex2_approx(m_ref - m_new);
          m_ref = m_new;
        } else if (m_new > m_ref + kRescaleLog2) {
          alpha_o = ex2_approx(m_ref - m_new);
          l *= alpha_o;
          m_ref = m_new;
          resc = true;
        }
      }
      }
      const float mr = (m_ref == -INFINITY) ? 0.f : m_ref;
      const uint64_t mr2 = f2_splat(mr);
      uint64_t rs2 = f2_splat(0.f);
      uint32_t pk[HC / 2];
#pragma unroll
      for (int e = 0; e < HC / 2; ++e) {
        float ya, yb;
        const uint64_t x2 = f2_pack(__uint_as_float(xr[2 * e]), __uint_as_float(xr[2 * e + 1]));
        f2_unpack(FIXM ? x2 : f2_sub(x2, mr2), ya, yb);
        const float p0 = ex2_approx(ya), p1 = ex2_approx(yb);
        const uint64_t p2 = f2_pack(p0, p1);
        rs2 = f2_add(rs2, p2);
        pk[e] = pack_bf16(p0, p1);
      }
      {
        float ra, rb;
        f2_unpack(rs2, ra, rb);
        l += ra + rb;
      }
      // P (bf16 pairs) over the first half of this thread's own score columns: the partner
      // warp may still be reading its half of S, so neither writes into the other's columns.
      const uint32_t pa = lane_addr + (uint32_t)((j & 1) * BN + half * HC);
#pragma unroll
      for (int c = 0; c < HC / 64; ++c) tmem_st32(pa + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + c * 32));
      if constexpr (HC / 2 == 16) tmem_st16(pa, pk);

      if (!FIXM && j >= 1) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, p.status));
      if (!FIXM && j >= 1 && __any_sync(0xffffffffu, resc)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = half * vcn; c < (half + 1) * vcn; ++c) {
          uint32_t orr[32];
          tmem_ld32(lane_addr + C::TM_O + c * 32, orr);
          tmem_wait_ld();
          reg_fence(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha_o);
          tmem_st32(lane_addr + C::TM_O + c * 32, orr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(j & 1));
      // a failed o_done wait travels to the partner in the next exchange
    }

    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, FIXM ? mbar_wait(o_fin, 0, p.status) : mbar_wait(o_done, (n - 1) & 1, p.status));
      tc_fence_after();
    }
    // Combine the two halves' sums (the running maxima already agree); slot 2 is used
    // only here.
    xbuf[(half * 3 + 2) * kBM + r] = l;
    pair_bar(wq);
    l += xbuf[((1 - half) * 3 + 2) * kBM + r];
    const bool has = l > 0.f;
    const float inv = has ? 1.f / l : 0.f;
    const float lse = has ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    if (ns > 1) {
      // Split partial: this split's normalised output (fp32) and its LSE, for the merge.
      const size_t prow = (((size_t)split * p.B + b) * p.Hq + h) * p.Sq + i;
      float *op = p.o_part + prow * D;
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t orr[32];
        if (n > 0) {
          tmem_ld32(lane_addr + C::TM_O + c * 32, orr);
          tmem_wait_ld();
          reg_fence(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if (row_ok) {
          float4 *dst = reinterpret_cast<float4 *>(op + c * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(orr[4 * v]) * inv, __uint_as_float(orr[4 * v + 1]) * inv,
                                 __uint_as_float(orr[4 * v + 2]) * inv, __uint_as_float(orr[4 * v + 3]) * inv);
        }
      }
      if (row_ok && half == 0) p.lse_part[prow] = lse;
    } else {
      __nv_bfloat16 *orow =
          static_cast<__nv_bfloat16 *>(p.O) + (((size_t)b * p.Sq + i) * p.Hq + h) * (C::WIDE ? p.D : D) + vc0 * 64;
#pragma unroll 1
      for (int c = half * vcn; c < (half + 1) * vcn; ++c) {
        uint32_t orr[32];
        if (n > 0) {
          tmem_ld32(lane_addr + C::TM_O + c * 32, orr);
          tmem_wait_ld();
          reg_fence(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if (row_ok) {
          uint32_t out[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            out[e] = pack_bf16(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(out[4 * v], out[4 * v + 1], out[4 * v + 2], out[4 * v + 3]);
        }
      }
      if (row_ok && half == 0 && vh == 0) p.LSE[((size_t)b * p.Hq + h) * p.Sq + i] = lse;
    }
  }

  __syncwarp();  // every warp reconverges (producer lanes leave their loops at different times)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int D, int BN, int NK, int NV>
cudaError_t launch_fwd(const Params &p, cudaStream_t st) {
  using C = FwdCfg<D, BN, NK, NV>;
  CUtensorMap tq, tk, tv;
  // The wide form reads the head dim at run time: whole 64-column chunks, above 256, at most D.
  if (C::WIDE && (p.D % 64 != 0 || p.D <= 256 || p.D > D)) return cudaErrorInvalidValue;
  const int Dm = C::WIDE ? p.D : D;
  if (!make_tmap_bshd(&tq, p.q, Dm, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb, kBM) ||
      !make_tmap_bshd(&tk, p.k, Dm, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, BN) ||
      !make_tmap_bshd(&tv, p.v, Dm, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb, C::HALF ? 64 : BN))
    return cudaErrorInvalidValue;
  if (C::WIDE && p.kv_splits > 1) return cudaErrorInvalidValue;  // the split-KV forward is not built for it
  auto kern = p.bias ? (p.cap <= 0.f                 ? fwd_tc_kernel<D, BN, NK, NV, false, false, true>
                        : p.cap <= kFixedMaxCap ? fwd_tc_kernel<D, BN, NK, NV, true, true, true>
                                                : fwd_tc_kernel<D, BN, NK, NV, true, false, true>)
                     : (p.cap <= 0.f                 ? fwd_tc_kernel<D, BN, NK, NV, false, false, false>
                        : p.cap <= kFixedMaxCap ? fwd_tc_kernel<D, BN, NK, NV, true, true, false>
                                                : fwd_tc_kernel<D, BN, NK, NV, true, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const long long nblk =
      (long long)((p.Sq + kBM - 1) / kBM) * p.Hq * p.B * (p.kv_splits > 1 ? p.kv_splits : 1) * (C::WIDE ? 2 : 1);
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidValue;
  Params q = p;
  if (!follow_work_list(nblk)) q.qorder = nullptr;
  kern<<<(unsigned)nblk, kThreads, C::SMEM, st>>>(tq, tk, tv, q);
  return counted(cudaGetLastError());
}

// Whether the grid fills two CTAs on every SM (the 64-key pair configuration); smaller grids --
// decode-like rows, split shares -- keep one CTA per SM on 128-key tiles, whose N = 128 score
// MMAs run at the full rate (decode-like workload forward 724 against 624 TFLOP/s).
bool pair_grid(const Params &p) {
  const long long nblk = (long long)((p.Sq + kBM - 1) / kBM) * p.Hq * p.B * (p.kv_splits > 1 ? p.kv_splits : 1);
  return nblk >= 2LL * device_sm_count();
}

}  // namespace

bool tc_supported(int D) { return D == 64 || D == 128 || D == 256 || (D > 256 && D <= 512 && D % 64 == 0); }

// Tiles.  Head dims 64 and 128, grids of at least two CTAs per SM: 64 keys per step, two-deep K
// and V rings, so that two score buffers and O take 256 TMEM columns and two CTAs share each
// SM -- one CTA's softmax warps overlap the other's MMAs and loads (measured against one CTA on
// 128-key tiles, same box: D=64 forward +20-22 %, D=128 +33 %; deeper rings changed nothing).
// Smaller grids: 128 keys per step, one CTA per SM.  Head dim 256: 128 keys per step
// (N = 128 score MMAs run at the full tensor rate, N = 64 ones at two thirds of it); two score
// buffers and O fill the 512 TMEM columns, and its 64 KiB K and V tiles leave room for one of
// each next to Q (measured 20 % faster than 64-key tiles with two-deep rings).  Head dims 320,
// 384, 448 and 512: the wide form.
cudaError_t tc_forward(const Params &p, cudaStream_t st) {
  switch (p.D) {
    case 64:
      return pair_grid(p) ? launch_fwd<64, 64, 2, 2>(p, st) : launch_fwd<64, 128, 4, 4>(p, st);
    case 128:
      return pair_grid(p) ? launch_fwd<128, 64, 2, 2>(p, st) : launch_fwd<128, 128, 3, 2>(p, st);
    case 256: return launch_fwd<256, 128, 1, 1>(p, st);
    case 320:
    case 384:
    case 448:
    case 512: return launch_fwd<512, 128, 2, 0>(p, st);  // wide form: two 32 KiB ring slots
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
