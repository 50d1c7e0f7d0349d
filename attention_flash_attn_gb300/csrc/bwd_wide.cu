// bwd_wide.cu -- tensor-core backward for bf16 with head dims 320, 384, 448 and 512.
//
// Above head dim 256 a CTA cannot hold the tensor-core backward's per-key-tile state: dK and dV
// of a 128-key tile alone need 1024 fp32 TMEM columns, and K and V tiles 256 KiB of shared
// memory (at 512).  The backward is therefore done in two steps, both on tcgen05 (the chunked head-dim
// accumulation above 256 named in the MaxText commit message quoted on tokamax PR #1121):
//
//   scores kernel: one CTA per 128-row query tile of one (batch, query head) and share of at
//     most four of its visible 128-key tiles.  Q stays in shared memory while S_j = Q K_j^T is
//     formed for each of those tiles j (K streamed
//     through a ring of 16 KiB slots, each a 64-column chunk of the tile); the softmax warps
//     write P = exp(t - LSE) and P f (f = 1 - tanh^2(u / cap), 1 without the cap) as bf16 into
//     scratch [B, Hq, Sq_pad, Sk_pad].  Then dO replaces Q and dP_j = dO V_j^T is formed for the
//     same tiles; dU = P f (dP - D) -- the gradient with respect to the pre-cap logits (tokamax
//     PR #1121, PR body: the factor is applied before dK and dbias) -- overwrites P f, and is
//     added into the dbias accumulator when there is a bias.
//   GEMM kernel: dV = sum over the group's query heads of P^T dO, dK = scale sum dU^T Q,
//     dQ = scale dU K -- one CTA per 128-row tile and part of the result's columns (of the
//     D / 64 column chunks, the first CTA takes ceil(D / 128), the second the rest), accumulated
//     in TMEM, operands by TMA, the contraction running over the visible range only.
//
// The head dim comes in whole 64-column chunks: a compile-time count for 512 (loop bounds and
// MMA shapes fixed: measured 6 % faster in the backward than the same code with a run-time
// count), read at run time for 320, 384 and 448; shared memory and TMEM are sized for 512.
//
// Work: 4 D flops per visible pair in the scores kernel (S, dP) and 6 D in the GEMMs (causal
// masks skip the zero blocks; windows and segments are multiplied through as zeros), against
// 10 D algorithmic.  Scratch: 2 B Hq Sq_pad Sk_pad bf16 values.
#include "../../include/attn_gb300.h"
#include "bwd_score.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;
using namespace bwd_score;

constexpr int kWD = 512;    // largest head dim (shared memory and TMEM are sized for it)
constexpr int kBM = 128;    // query rows per scores CTA, result rows per GEMM CTA
constexpr int kBN = 128;    // keys per tile
constexpr int kNR = 4;      // ring slots of the scores kernel
constexpr int kSlot = kBN * 128;       // 16 KiB: one 64-column chunk of a 128-row tile
constexpr int kQBytes = kBM * kWD * 2; // 128 KiB at most

// ---------------------------------------------------------------------------- scores kernel

struct ScoresCfg {
  static constexpr int OFF_Q = 0;                      // Q, then dO
  static constexpr int OFF_R = kQBytes;                // ring
  static constexpr int OFF_BAR = OFF_R + kNR * kSlot;
  static constexpr int NBAR = 3 + 2 * kNR + 4;         // q_full, do_full, q_free, ring, s_full x2, p_free x2
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};
constexpr int kScoresThreads = 320;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 element-wise
constexpr int kScoresChunk = 4;      // key tiles per scores CTA at most

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int e = 0; e < N; ++e) asm volatile("" : "+r"(r[e]));
}

// Scratch rows: element (b, h, i, j) at ((b Hq + h) sq_pad + i) sk_pad + j.
struct WideScratch {
  __nv_bfloat16 *P, *U;  // P, then P f / dU
  int sq_pad, sk_pad;
};

// NCHT: the head dim's 64-column chunks when fixed at compile time (8), else 0 (read from p.D).
template <bool CAP, bool BIAS, int NCHT>
__global__ void __launch_bounds__(kScoresThreads, 1)
    wide_scores_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const Params p, const WideScratch w) {
  using C = ScoresCfg;
  constexpr int HC = kBN / 2;  // key columns per element-wise thread and tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *misc_i = reinterpret_cast<int *>(smem + C::OFF_MISC);
  {  // A wait elsewhere already gave up: do nothing.
    if (threadIdx.x == 0) misc_i[12] = (status_peek(p.status) & kStatusWaitTimeout) ? 1 : 0;
    __syncthreads();
    if (misc_i[12]) return;
  }

  // Grid: query tile slowest (latest, heaviest under causal masks, first), then batch, head, and
  // the share of the visible key tiles (at most kScoresChunk each; P and dU of a pair depend on
  // that pair alone, so the key range splits freely).
  const int nqt = (p.Sq + kBM - 1) / kBM;
  const int nks = (p.Sk + kBN * kScoresChunk - 1) / (kBN * kScoresChunk);
  const int ks = (int)(blockIdx.x % (unsigned)nks);
  const unsigned bx = blockIdx.x / (unsigned)nks;
  const int bh = (int)(bx % (unsigned)(p.Hq * p.B));
  const int qt = nqt - 1 - (int)(bx / (unsigned)(p.Hq * p.B));
  const int h = bh % p.Hq, b = bh / p.Hq, g = h / p.G;
  const int i0 = qt * kBM, i1 = min(i0 + kBM, p.Sq) - 1;
  const int off = p.Sk - p.Sq;
  const int nch = NCHT > 0 ? NCHT : p.D / 64;  // 64-column chunks of the head dim

  // Keys this query tile can see (uniform across the CTA).
  int klo = 0, khi = p.Sk;
  if (!p.qoff) {
    if (p.window > 0) klo = max(klo, i0 + off - p.window + 1);
    if (p.causal) khi = min(khi, i1 + off + 1);
  }
  if (p.qtile) {
    const int4 c = p.qtile[(size_t)b * nqt + qt];
    klo = max(klo, c.x);
    khi = min(khi, c.y);
  }
  const int tv0 = klo / kBN;
  const int nv = (klo < khi) ? (khi + kBN - 1) / kBN - tv0 : 0;
  const int t0 = tv0 + ks * kScoresChunk;                     // this CTA's share of the tiles
  const int n = max(0, min(nv - ks * kScoresChunk, kScoresChunk));
  if (n == 0) return;  // nothing to write: the scratch was zeroed

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0, do_full = bar0 + 8u, q_free = bar0 + 16u;
  auto r_full = [&](int s) { return bar0 + 8u * (3 + s); };
  auto r_empty = [&](int s) { return bar0 + 8u * (3 + kNR + s); };
  auto s_full = [&](int x) { return bar0 + 8u * (3 + 2 * kNR + x); };
  auto p_free = [&](int x) { return bar0 + 8u * (5 + 2 * kNR + x); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *red = misc_i + 4;  // [8]

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(do_full, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < kNR; ++s) {
      mbar_init(r_full(s), 1);
      mbar_init(r_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_free(x), 256);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0 && (tmem & 0xFFFFu) + 256 > 512) set_status(p.status, kStatusBadTmemAlloc);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Q, K_0 .. K_{n-1}; once every S MMA has read Q, dO into its place; V_0 .. V_{n-1}.
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(q_full, nch * (kBM * 128));
#pragma unroll 1
      for (int c = 0; c < nch; ++c)
        tma_load_4d(sbase + C::OFF_Q + c * (kBM * 128), &tmQ, q_full, c * 64, i0, h, b);
      int u = 0;
      auto slot_load = [&](const CUtensorMap *tm, int d0, int row) -> bool {
        const int s = u % kNR;
        if (u >= kNR && !mbar_wait(r_empty(s), ((u / kNR) - 1) & 1, p.status)) return false;
        mbar_arrive_expect_tx(r_full(s), kSlot);
        tma_load_4d(sbase + C::OFF_R + s * kSlot, tm, r_full(s), d0, row, g, b);
        ++u;
        return true;
      };
      bool okp = true;
      for (int j = 0; okp && j < n; ++j)
        for (int c = 0; okp && c < nch; ++c) okp = slot_load(&tmK, c * 64, (t0 + j) * kBN);
      if (okp && mbar_wait(q_free, 0, p.status)) {
        mbar_arrive_expect_tx(do_full, nch * (kBM * 128));
#pragma unroll 1
        for (int c = 0; c < nch; ++c)
          tma_load_4d(sbase + C::OFF_Q + c * (kBM * 128), &tmdO, do_full, c * 64, i0, h, b);
        for (int j = 0; okp && j < n; ++j)
          for (int c = 0; okp && c < nch; ++c) okp = slot_load(&tmV, c * 64, (t0 + j) * kBN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Tile jj < n: S_jj = Q K_jj^T; jj >= n: dP_{jj-n} = dO V_{jj-n}^T; into score buffer jj & 1
    // once the element-wise warps have copied out tile jj - 2.
    if (n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      const uint64_t dq0 = sw128_desc(sbase + C::OFF_Q, 16, 1024);
      int u = 0;
      bool ok = mbar_wait_warp(q_full, 0, p.status);
      for (int jj = 0; ok && jj < 2 * n; ++jj) {
        if (jj == n && !mbar_wait_warp(do_full, 0, p.status)) break;
        const int x = jj & 1;
        if (jj >= 2 && !mbar_wait_warp(p_free(x), ((jj - 2) >> 1) & 1, p.status)) break;
        tc_fence_after();
        const uint32_t dS = tmem + (uint32_t)(x * kBN);
#pragma unroll 1
        for (int c = 0; c < nch; ++c, ++u) {
          const int s = u % kNR;
          if (!mbar_wait_warp(r_full(s), (u / kNR) & 1, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t qd = desc_at(dq0, c * (kBM * 128));
          const uint64_t kd = sw128_desc(sbase + C::OFF_R + s * kSlot, 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) mma_ss_w(dS, desc_at(qd, k4 * 32), desc_at(kd, k4 * 32), idS, (c | k4) != 0);
          mma_commit_w(r_empty(s));
        }
        if (!ok) break;
        mma_commit_w(s_full(x));
        if (jj == n - 1) mma_commit_w(q_free);  // every S MMA has read Q
      }
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;
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
    if (!row_ok) {
      lo = 0;
      hi = 0;
    }
    const bool any_pairwise = p.seg_q != nullptr && !p.seg_mono[b];
    const size_t rowi = ((size_t)b * p.Hq + h) * w.sq_pad + (row_ok ? i : 0);
    const float lse2 = row_ok ? p.lse2p[((size_t)b * p.Hq + h) * p.sq_pad + i] : INFINITY;
    const float dvec = row_ok ? p.Dvec[((size_t)b * p.Hq + h) * p.sq_pad + i] : 0.f;
    __nv_bfloat16 *prow = w.P + rowi * w.sk_pad;
    __nv_bfloat16 *urow = w.U + rowi * w.sk_pad;
    const unsigned short *brow =
        BIAS ? static_cast<const unsigned short *>(p.bias) + (size_t)b * p.bias_sb + (size_t)h * p.bias_sh +
                   (size_t)min(i, p.Sq - 1) * p.Sk
             : nullptr;
    float *dbrow = BIAS ? p.dbias_acc + (((size_t)(p.bias_B == 1 ? 0 : b) * p.bias_H + (p.bias_H == 1 ? 0 : h)) *
                                             p.Sq + min(i, p.Sq - 1)) * p.Sk
                        : nullptr;
    const BwdScore ks(p.scale, p.inv_cap, p.cap);
    const uint64_t lse2x2 = f2_splat(lse2), dx2 = f2_splat(dvec);
    bool ok = true;

    for (int jj = 0; ok && jj < 2 * n; ++jj) {
      const int x = jj & 1;
      const int j = jj < n ? jj : jj - n;
      const int j0 = (t0 + j) * kBN + half * HC;  // this thread's first key column
      const bool sweep1 = jj < n;
      uint32_t aux[HC / 2];  // sweep 1: bias pairs; sweep 2: P f pairs
      if (sweep1) {
        if constexpr (BIAS) {
#pragma unroll
          for (int e = 0; e < HC / 2; ++e) {
            const int ja = j0 + 2 * e;
            const uint32_t a = __ldg(brow + min(ja, p.Sk - 1)), c = __ldg(brow + min(ja + 1, p.Sk - 1));
            aux[e] = (ja < p.Sk ? a : 0u) | (ja + 1 < p.Sk ? c << 16 : 0u);
          }
        }
      } else if (row_ok) {
        const uint4 *src = reinterpret_cast<const uint4 *>(urow + j0);
#pragma unroll
        for (int v = 0; v < HC / 8; ++v) {
          const uint4 y = src[v];
          aux[4 * v] = y.x;
          aux[4 * v + 1] = y.y;
          aux[4 * v + 2] = y.z;
          aux[4 * v + 3] = y.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < HC / 2; ++e) aux[e] = 0u;
      }
      const bool got = __all_sync(0xffffffffu, mbar_wait(s_full(x), (jj >> 1) & 1, p.status));
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t xr[HC];
#pragma unroll
      for (int c = 0; c < HC / 32; ++c)
        tmem_ld32(lane_addr + (uint32_t)(x * kBN + half * HC + c * 32), *reinterpret_cast<uint32_t(*)[32]>(xr + c * 32));
      tmem_wait_ld();
      reg_fence(xr);
      tc_fence_before();
      mbar_arrive(p_free(x));  // the score buffer may be overwritten

      // Visibility of this thread's columns: every column of a tile inside [lo, hi) with sorted
      // ids, else column by column.
      const bool full = !any_pairwise && j0 >= lo && j0 + HC <= hi;
      uint32_t o1[HC / 2], o2[HC / 2];
#pragma unroll
      for (int e = 0; e < HC / 2; ++e) {
        const int ja = j0 + 2 * e;
        bool va = true, vb = true;
        if (!full) {
          va = ja >= lo && ja < hi;
          vb = ja + 1 >= lo && ja + 1 < hi;
          if (seg_pairwise) {
            va = va && __ldg(segk + min(ja, p.Sk - 1)) == sid;
            vb = vb && __ldg(segk + min(ja + 1, p.Sk - 1)) == sid;
          }
        }
        if (sweep1) {
          uint64_t y, f;
          score_pair<CAP, true, true>(xr[2 * e], xr[2 * e + 1], lse2x2, ks, y, f,
                                      BIAS ? bias_pair(aux[e]) : f2_splat(0.f));
          float pa, pb, fa, fb;
          f2_unpack(ex2_pair(y), pa, pb);
          f2_unpack(f, fa, fb);
          pa = va ? pa : 0.f;
          pb = vb ? pb : 0.f;
          o1[e] = pack_bf16(pa, pb);
          o2[e] = pack_bf16(pa * fa, pb * fb);
        } else {
          // dU = P f (dP - D): the gradient with respect to the pre-cap logit (and the bias)
          const uint64_t pf = bias_pair(aux[e]);
          const uint64_t dp = f2_pack(__uint_as_float(xr[2 * e]), __uint_as_float(xr[2 * e + 1]));
          float ua, ub;
          f2_unpack(f2_mul(pf, f2_sub(dp, dx2)), ua, ub);
          ua = va ? ua : 0.f;
          ub = vb ? ub : 0.f;
          if constexpr (BIAS) {
            red_add_f32_if(dbrow + min(ja, p.Sk - 1), ua, (va && row_ok) ? 1u : 0u);
            red_add_f32_if(dbrow + min(ja + 1, p.Sk - 1), ub, (vb && row_ok) ? 1u : 0u);
          }
          o2[e] = pack_bf16(ua, ub);
        }
      }
      if (row_ok) {
        uint4 *d2 = reinterpret_cast<uint4 *>(urow + j0);
#pragma unroll
        for (int v = 0; v < HC / 8; ++v) d2[v] = make_uint4(o2[4 * v], o2[4 * v + 1], o2[4 * v + 2], o2[4 * v + 3]);
        if (sweep1) {
          uint4 *d1 = reinterpret_cast<uint4 *>(prow + j0);
#pragma unroll
          for (int v = 0; v < HC / 8; ++v) d1[v] = make_uint4(o1[4 * v], o1[4 * v + 1], o1[4 * v + 2], o1[4 * v + 3]);
        }
      }
    }
    (void)red;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------- GEMM kernel
//
// C[m, n] = alpha sum_z sum_k A_z[m, k] B_z[k, n] for one 128-row tile m0 .. m0 + 127 and one
// part of the head dim's columns (two CTAs per row tile; at most 256 columns each), in three
// forms:
//   DV: m = key, k = query, z = the query heads of the kv group: A = P^T, B = dO;  alpha = 1
//   DK: the same with A = dU^T, B = Q;                                            alpha = scale
//   DQ: m = query, k = key, z = the query head itself: A = dU, B = K;             alpha = scale
// A comes from the [B, Hq, Sq_pad, Sk_pad] scratch (key index contiguous): M-major for DV / DK,
// K-major for DQ.  B is a bshd tensor with the head dim contiguous (N-major).  The contraction
// runs over 64-row steps of the range that causal / window masks leave visible to the tile.
enum { kGemmDV = 0, kGemmDK = 1, kGemmDQ = 2 };
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kKStep = 64;
constexpr int kNHalf = kWD / 2;               // result columns per CTA, at most
constexpr int kABytes = kBM * kKStep * 2;     // 16 KiB
constexpr int kBBytes = kKStep * kNHalf * 2;  // 32 KiB
constexpr int kGStages = 4;
struct GemmCfg {
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = kGStages * kABytes;
  static constexpr int OFF_BAR = OFF_B + kGStages * kBBytes;
  static constexpr int NBAR = 2 * kGStages + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// NCHT: as for the scores kernel.
template <int MODE, int NCHT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    wide_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p,
                     __nv_bfloat16 *out, float alpha) {
  using C = GemmCfg;
  constexpr bool A_MN = MODE != kGemmDQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *misc_i = reinterpret_cast<int *>(smem + C::OFF_MISC);
  {
    if (threadIdx.x == 0) misc_i[12] = (status_peek(p.status) & kStatusWaitTimeout) ? 1 : 0;
    __syncthreads();
    if (misc_i[12]) return;
  }
  // Grid: (result tile and column half, head or kv group, batch).
  const int mt = blockIdx.x >> 1, nh = blockIdx.x & 1, hz = blockIdx.y, b = blockIdx.z;
  // This CTA's 64-column chunks of the result: nb of them from chunk cb.
  const int nch = NCHT > 0 ? NCHT : p.D / 64;
  const int cb = nh == 0 ? 0 : (nch + 1) / 2, nb = nh == 0 ? (nch + 1) / 2 : nch / 2;
  const int M = MODE == kGemmDQ ? p.Sq : p.Sk;
  const int m0 = mt * kBM, m1 = min(m0 + kBM, M) - 1;
  const int nz = MODE == kGemmDQ ? 1 : p.G;
  const int Klen = MODE == kGemmDQ ? p.Sk : p.Sq;
  const int off = p.Sk - p.Sq;
  // Contraction range visible to the tile (one offset for the whole matrix; with per-sequence
  // offsets the whole range).
  int klo = 0, khi = Klen;
  if (!p.qoff) {
    if (MODE == kGemmDQ) {  // keys seen by queries m0 .. m1
      if (p.causal) khi = min(khi, m1 + off + 1);
      if (p.window > 0) klo = max(klo, m0 + off - p.window + 1);
    } else {                // queries that see keys m0 .. m1
      if (p.causal) klo = max(klo, m0 - off);
      if (p.window > 0) khi = min(khi, m1 - off + p.window);
    }
  }
  const int s0 = max(klo, 0) / kKStep;
  const int nsteps = khi > klo ? (khi + kKStep - 1) / kKStep - s0 : 0;
  const int total = nsteps * nz;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto f_full = [&](int s) { return bar0 + 8u * s; };
  auto f_empty = [&](int s) { return bar0 + 8u * (kGStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kGStages);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(f_full(s), 1);
      mbar_init(f_empty(s), 1);
    }
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kNHalf);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0 && (tmem & 0xFFFFu) + kNHalf > 512) set_status(p.status, kStatusBadTmemAlloc);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && total > 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      for (int it = 0; it < total; ++it) {
        const int z = it / nsteps, ks = s0 + it % nsteps;
        const int s = it % kGStages;
        if (it >= kGStages && !mbar_wait(f_empty(s), ((it / kGStages) - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(f_full(s), kABytes + nb * (kKStep * 128));
        const uint32_t a_dst = sbase + C::OFF_A + s * kABytes, b_dst = sbase + C::OFF_B + s * kBBytes;
        const int k0 = ks * kKStep;
        if constexpr (MODE == kGemmDQ) {
          // A = dU [queries m, keys k]: one box of 64 keys x 128 queries (K-major)
          tma_load_4d(a_dst, &tmA, f_full(s), k0, m0, hz, b);
#pragma unroll 4
          for (int c = 0; c < nb; ++c)  // B = K_g [keys k, this CTA's columns of d]
            tma_load_4d(b_dst + c * (kKStep * 128), &tmB, f_full(s), (cb + c) * 64, k0, hz / p.G, b);
        } else {
          const int h = hz * p.G + z;
          // A = P^T or dU^T: two boxes of 64 keys (m) x 64 queries (k), keys contiguous (M-major)
          tma_load_4d(a_dst, &tmA, f_full(s), m0, k0, h, b);
          tma_load_4d(a_dst + kKStep * 128, &tmA, f_full(s), m0 + 64, k0, h, b);
#pragma unroll 4
          for (int c = 0; c < nb; ++c)  // B = dO_h or Q_h [queries k, this CTA's columns of d]
            tma_load_4d(b_dst + c * (kKStep * 128), &tmB, f_full(s), (cb + c) * 64, k0, h, b);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idC = idesc_bf16(kBM, nb * 64, A_MN, true);
    bool ok = true;
    for (int it = 0; ok && it < total; ++it) {
      const int s = it % kGStages;
      if (!mbar_wait_warp(f_full(s), (it / kGStages) & 1, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint64_t da = A_MN ? sw128_desc(sbase + C::OFF_A + s * kABytes, kKStep * 128, 1024)
                               : sw128_desc(sbase + C::OFF_A + s * kABytes, 16, 1024);
      const uint64_t db = sw128_desc(sbase + C::OFF_B + s * kBBytes, kKStep * 128, 1024);
#pragma unroll
      for (int k4 = 0; k4 < kKStep / 16; ++k4)
        mma_ss_w(tmem, desc_at(da, A_MN ? k4 * 2048 : k4 * 32), desc_at(db, k4 * 2048), idC,
                 (it > 0 || k4 > 0) ? 1u : 0u);
      mma_commit_w(f_empty(s));
    }
    mma_commit_w(acc_full);  // every MMA of this CTA has completed (or none was issued)
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int m = m0 + row;
    const bool have = total > 0;
    bool ok = true;
    if (have) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.status));
    tc_fence_after();
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    __nv_bfloat16 *dst = out + (MODE == kGemmDQ ? (((size_t)b * p.Sq + min(m, M - 1)) * p.Hq + hz) * p.D
                                                : (((size_t)b * p.Sk + min(m, M - 1)) * p.Hkv + hz) * p.D) +
                         cb * 64;
#pragma unroll 1
    for (int c = 0; c < 2 * nb; ++c) {
      uint32_t v[32];
      if (have && ok) {
        tmem_ld32(lane_addr + c * 32, v);
        tmem_wait_ld();
        reg_fence(v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      if (m <= m1) {
        uint4 *d = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          d[q] = make_uint4(pack_bf16(__uint_as_float(v[8 * q]) * alpha, __uint_as_float(v[8 * q + 1]) * alpha),
                            pack_bf16(__uint_as_float(v[8 * q + 2]) * alpha, __uint_as_float(v[8 * q + 3]) * alpha),
                            pack_bf16(__uint_as_float(v[8 * q + 4]) * alpha, __uint_as_float(v[8 * q + 5]) * alpha),
                            pack_bf16(__uint_as_float(v[8 * q + 6]) * alpha, __uint_as_float(v[8 * q + 7]) * alpha));
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kNHalf);
  }
}

template <int MODE>
cudaError_t launch_gemm(const Params &p, const CUtensorMap &ta, const CUtensorMap &tb, __nv_bfloat16 *out,
                        float alpha, cudaStream_t st) {
  auto kern = p.D == kWD ? wide_gemm_kernel<MODE, kWD / 64> : wide_gemm_kernel<MODE, 0>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::SMEM);
  if (e != cudaSuccess) return e;
  const int M = MODE == kGemmDQ ? p.Sq : p.Sk;
  const dim3 grid(2 * ((M + kBM - 1) / kBM), MODE == kGemmDQ ? p.Hq : p.Hkv, p.B);
  kern<<<grid, kGemmThreads, GemmCfg::SMEM, st>>>(ta, tb, p, out, alpha);
  return counted(cudaGetLastError());
}

}  // namespace

size_t wide_bwd_scratch_bytes(int B, int Hq, int Sq, int Sk) {
  const size_t sq_pad = (size_t)(Sq + 127) / 128 * 128, sk_pad = (size_t)(Sk + 127) / 128 * 128;
  return 2 * (size_t)B * Hq * sq_pad * sk_pad * sizeof(__nv_bfloat16);
}

cudaError_t wide_backward(const Params &p, void *scratch, cudaStream_t st) {
  if (p.D % 64 != 0 || p.D <= 256 || p.D > kWD || p.B > 65535 || p.Hq > 65535) return cudaErrorInvalidValue;
  const int D = p.D;
  WideScratch w;
  w.sq_pad = (p.Sq + 127) / 128 * 128;
  w.sk_pad = (p.Sk + 127) / 128 * 128;
  const size_t plane = (size_t)p.B * p.Hq * w.sq_pad * w.sk_pad;
  w.P = static_cast<__nv_bfloat16 *>(scratch);
  w.U = w.P + plane;
  // Blocks the scores kernel does not visit (no visible pair) must read as zero in the GEMMs.
  cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * plane * sizeof(__nv_bfloat16), st);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tdo, tk, tv, tp, tu_mn, tu_k, tdo_b, tq_b, tk_b;
  const long long ss = w.sk_pad, sh = (long long)w.sq_pad * w.sk_pad, sb = sh * p.Hq;
  if (!make_tmap_bshd(&tq, p.q, D, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb, kBM) ||
      !make_tmap_bshd(&tdo, p.dO, D, p.Sq, p.Hq, p.B, (long long)p.Hq * D, D, (long long)p.Sq * p.Hq * D,
                      kBM) ||
      !make_tmap_bshd(&tk, p.k, D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, kBN) ||
      !make_tmap_bshd(&tv, p.v, D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb, kBN) ||
      // scratch planes as (key, query, head, batch): 64 x 64 boxes (M-major A of dV / dK) and
      // 64 keys x 128 queries (K-major A of dQ)
      !make_tmap_bshd(&tp, w.P, w.sk_pad, w.sq_pad, p.Hq, p.B, ss, sh, sb, kKStep) ||
      !make_tmap_bshd(&tu_mn, w.U, w.sk_pad, w.sq_pad, p.Hq, p.B, ss, sh, sb, kKStep) ||
      !make_tmap_bshd(&tu_k, w.U, w.sk_pad, w.sq_pad, p.Hq, p.B, ss, sh, sb, kBM) ||
      // B operands: 64-row boxes of dO, Q, K
      !make_tmap_bshd(&tdo_b, p.dO, D, p.Sq, p.Hq, p.B, (long long)p.Hq * D, D, (long long)p.Sq * p.Hq * D,
                      kKStep) ||
      !make_tmap_bshd(&tq_b, p.q, D, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb, kKStep) ||
      !make_tmap_bshd(&tk_b, p.k, D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, kKStep))
    return cudaErrorInvalidValue;
  const bool fixed = D == kWD;
  auto kern = p.bias ? (p.cap > 0.f ? (fixed ? wide_scores_kernel<true, true, kWD / 64> : wide_scores_kernel<true, true, 0>)
                                    : (fixed ? wide_scores_kernel<false, true, kWD / 64> : wide_scores_kernel<false, true, 0>))
                     : (p.cap > 0.f ? (fixed ? wide_scores_kernel<true, false, kWD / 64> : wide_scores_kernel<true, false, 0>)
                                    : (fixed ? wide_scores_kernel<false, false, kWD / 64> : wide_scores_kernel<false, false, 0>));
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ScoresCfg::SMEM);
  if (e != cudaSuccess) return e;
  const long long nks = (p.Sk + kBN * kScoresChunk - 1) / (kBN * kScoresChunk);
  const long long nblk = (long long)((p.Sq + kBM - 1) / kBM) * p.Hq * p.B * nks;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<(unsigned)nblk, kScoresThreads, ScoresCfg::SMEM, st>>>(tq, tdo, tk, tv, p, w);
  if ((e = counted(cudaGetLastError())) != cudaSuccess) return e;
  __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(p.dQ), *dk = static_cast<__nv_bfloat16 *>(p.dK),
                *dv = static_cast<__nv_bfloat16 *>(p.dV);
  if ((e = launch_gemm<kGemmDV>(p, tp, tdo_b, dv, 1.f, st)) != cudaSuccess) return e;
  if ((e = launch_gemm<kGemmDK>(p, tu_mn, tq_b, dk, p.scale, st)) != cudaSuccess) return e;
  return launch_gemm<kGemmDQ>(p, tu_k, tk_b, dq, p.scale, st);
}

}  // namespace attn
