// api.cu -- the C ABI declared in include/attn_gb300.h: argument validation (fail closed:
// an invalid or unsupported request never launches anything), workspace layout, and the
// launch sequence of the forward and backward passes on the caller's stream.
#include <math.h>
#include <algorithm>
#include <stdint.h>
#include <string.h>

#include "../../include/attn_gb300.h"
#include "common.cuh"
#include "internal.h"

namespace attn {

std::atomic<unsigned long long> g_launches{0};

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Mask metadata carve-up (segment / cu_seqlens calls), relative to the start of its region:
// a caller's buffer from attn_meta_build, or a region of the workspace.  [0, 256) holds a
// status area of its own (used by attn_meta_build).  Offsets are 0 when a region is absent.
struct MetaLayout {
  size_t mono = 0, qrange = 0, krange = 0, qrun = 0, krun = 0, seg = 0, segk = 0, qoff = 0, koff = 0;
  size_t qtile = 0, ktile = 0, qwork = 0, kwork = 0, qorder = 0, korder = 0;
  size_t total = 0;  // 0: the call needs no metadata
};

// Workspace carve-up.  Offsets are 0 when a region is absent.
struct Layout {
  size_t meta = 0;  // the metadata region, when the call needs one and args->meta is NULL
  size_t dvec = 0, lse2 = 0, dsplit = 0, dsink_part = 0, dqacc = 0, dbias_acc = 0, wide = 0;
  size_t o_part = 0, lse_part = 0;
  size_t total = 0;
};

bool use_tc(const attn_args *a) { return a->dtype == ATTN_DTYPE_BF16 && a->Sk > 0 && tc_supported(a->D); }
bool use_tc_bwd(const attn_args *a) { return use_tc(a) && tc_bwd_supported(a->D); }
// Head dims 320 .. 512 (the wide form): the scores-plus-GEMMs backward, while its two scratch
// planes stay within 16 GiB (longer rows fall back to the FFMA kernels).
constexpr size_t kWideScratchMax = size_t(16) << 30;
bool use_wide_bwd(const attn_args *a) {
  return use_tc(a) && a->D > 256 && wide_bwd_scratch_bytes(a->B, a->Hq, a->Sq, a->Sk) <= kWideScratchMax;
}

constexpr int kMaxKvSplits = 64;
// The split-KV forward applies to the tensor-core path only, head dims up to 256.
bool split_kv(const attn_args *a) { return a->kv_splits > 1 && use_tc(a) && a->D <= 256; }

size_t dbias_elems(const attn_args *a) {
  if (!a->bias) return 0;
  const size_t bb = a->bias_stride_b ? (size_t)a->B : 1, hb = a->bias_stride_h ? (size_t)a->Hq : 1;
  return bb * hb * (size_t)a->Sq * (size_t)a->Sk;
}

bool needs_meta(const attn_args *a) { return (a->seg_q || a->cu_seqlens) && a->B > 0; }

// Whether the work lists are built: at most work_order_max_tiles() tiles per axis.
bool work_lists(const attn_args *a) {
  const long long nq = (long long)a->B * ((a->Sq + 127) / 128), nk = (long long)a->B * ((a->Sk + 127) / 128);
  return nq <= work_order_max_tiles() && nk <= work_order_max_tiles();
}

MetaLayout meta_layout(const attn_args *a) {
  MetaLayout M;
  if (!needs_meta(a)) return M;
  size_t off = kAlign;  // [0, 256): status area of a standalone metadata buffer
  const size_t nq = (a->Sq + 63) / 64, nk = (a->Sk + 63) / 64;
  const size_t nq128 = (a->Sq + 127) / 128, nk128 = (a->Sk + 127) / 128;
  M.mono = off; off += align_up((size_t)a->B);
  M.qrange = off; off += align_up((size_t)a->B * nq * sizeof(int2));
  M.krange = off; off += align_up((size_t)a->B * nk * sizeof(int2));
  M.qrun = off; off += align_up((size_t)a->B * a->Sq * sizeof(int2));
  M.krun = off; off += align_up((size_t)a->B * a->Sk * sizeof(int2));
  if (a->cu_seqlens) { M.seg = off; off += align_up((size_t)a->Sq * sizeof(int)); }
  if (a->cu_seqlens_k) {
    M.segk = off; off += align_up((size_t)a->Sk * sizeof(int));
    M.qoff = off; off += align_up((size_t)a->Sq * sizeof(int));
    M.koff = off; off += align_up((size_t)a->Sk * sizeof(int));
  }
  M.qtile = off; off += align_up((size_t)a->B * nq128 * sizeof(int4));
  M.ktile = off; off += align_up((size_t)a->B * nk128 * sizeof(int4));
  M.qwork = off; off += align_up((size_t)a->B * nq128 * sizeof(long long));
  M.kwork = off; off += align_up((size_t)a->B * nk128 * sizeof(long long));
  if (work_lists(a)) {
    M.qorder = off; off += align_up((size_t)a->B * nq128 * sizeof(int2));
    M.korder = off; off += align_up((size_t)a->B * nk128 * sizeof(int2));
  }
  M.total = off;
  return M;
}

Layout layout(const attn_args *a, bool bwd) {
  Layout L;
  size_t off = kAlign;  // [0, 256): status word
  if (needs_meta(a) && !a->meta) {
    L.meta = off;
    off += meta_layout(a).total;
  }
  if (!bwd && split_kv(a)) {
    const size_t rows = (size_t)a->kv_splits * a->B * a->Hq * a->Sq;
    L.o_part = off; off += align_up(rows * a->D * sizeof(float));
    L.lse_part = off; off += align_up(rows * sizeof(float));
  }
  if (bwd) {
    const size_t sq_pad = (size_t)(a->Sq + 127) / 128 * 128;
    L.dvec = off; off += align_up((size_t)a->B * a->Hq * sq_pad * sizeof(float));
    if (use_tc_bwd(a) || use_wide_bwd(a)) { L.lse2 = off; off += align_up((size_t)a->B * a->Hq * sq_pad * sizeof(float)); }
    if (use_tc_bwd(a) && tc_bwd_fused(a->D)) { L.dsplit = off; off += align_up((size_t)a->B * a->Hq * sq_pad * 16); }
    if (a->sink) {
      L.dsink_part = off;
      off += align_up((size_t)a->Hq * bwd_pre_partials_max(a->B, a->Sq) * sizeof(float));
    }
    if (use_tc_bwd(a)) { L.dqacc = off; off += align_up((size_t)a->B * a->Sq * a->Hq * a->D * sizeof(float)); }
    if (a->bias) { L.dbias_acc = off; off += align_up(dbias_elems(a) * sizeof(float)); }
    if (use_wide_bwd(a)) { L.wide = off; off += align_up(wide_bwd_scratch_bytes(a->B, a->Hq, a->Sq, a->Sk)); }
  }
  L.total = off;
  return L;
}

int validate(const attn_args *a) {
  if (!a) return ATTN_ERR_INVALID;
  if (a->dtype != ATTN_DTYPE_BF16 && a->dtype != ATTN_DTYPE_F32) return ATTN_ERR_INVALID;
  if (a->B < 0 || a->Sq < 0 || a->Sk < 0 || a->Hq < 1 || a->Hkv < 1 || a->D < 1) return ATTN_ERR_INVALID;
  if (a->Hq % a->Hkv != 0) return ATTN_ERR_INVALID;
  if (a->D % 8 != 0) return ATTN_ERR_INVALID;
  if (a->D > 512) return ATTN_ERR_UNSUPPORTED;
  if (!isfinite(a->scale)) return ATTN_ERR_INVALID;
  if (!isfinite(a->softcap) || a->softcap < 0.f) return ATTN_ERR_INVALID;
  if (a->B > 0 && a->Sq > 0 && !a->q) return ATTN_ERR_INVALID;
  if (a->B > 0 && a->Sk > 0 && (!a->k || !a->v)) return ATTN_ERR_INVALID;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v)) return ATTN_ERR_INVALID;
  const int64_t vec = a->dtype == ATTN_DTYPE_BF16 ? 8 : 4;  // elements per 16 bytes
  const int64_t st[9] = {a->q_stride_b, a->q_stride_s, a->q_stride_h, a->k_stride_b, a->k_stride_s,
                         a->k_stride_h, a->v_stride_b, a->v_stride_s, a->v_stride_h};
  for (int64_t s : st)
    if (s < 0 || s % vec != 0) return ATTN_ERR_INVALID;
  if (a->Sq > 0 && a->q_stride_s < (int64_t)a->D) return ATTN_ERR_INVALID;
  if (a->bias) {
    if (a->bias_stride_b < 0 || a->bias_stride_h < 0 || !aligned16(a->bias)) return ATTN_ERR_INVALID;
  }
  if ((a->seg_q == nullptr) != (a->seg_k == nullptr)) return ATTN_ERR_INVALID;
  if (a->softmax_type != ATTN_SOFTMAX_DEFAULT && a->softmax_type != ATTN_SOFTMAX_OFF_BY_ONE) return ATTN_ERR_INVALID;
  if (a->softmax_type == ATTN_SOFTMAX_OFF_BY_ONE && a->sink) return ATTN_ERR_INVALID;
  if (a->kv_splits < 0 || a->kv_splits > kMaxKvSplits) return ATTN_ERR_INVALID;
  if (a->cu_seqlens) {
    if (a->seg_q) return ATTN_ERR_UNSUPPORTED;
    if (a->B != 1 || a->nseq < 0) return ATTN_ERR_INVALID;
    if (!a->cu_seqlens_k && a->Sq != a->Sk) return ATTN_ERR_INVALID;
  } else if (a->cu_seqlens_k) {
    return ATTN_ERR_INVALID;
  }
  if (((uintptr_t)a->meta % kAlign) != 0) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

// Points the parameter block's metadata fields into a metadata region at `m`.
void set_meta(const attn_args *a, char *m, Params &p) {
  const MetaLayout M = meta_layout(a);
  p.seg_mono = reinterpret_cast<unsigned char *>(m + M.mono);
  p.qrange = reinterpret_cast<int2 *>(m + M.qrange);
  p.krange = reinterpret_cast<int2 *>(m + M.krange);
  p.qrun = reinterpret_cast<int2 *>(m + M.qrun);
  p.krun = reinterpret_cast<int2 *>(m + M.krun);
  p.qtile = reinterpret_cast<int4 *>(m + M.qtile);
  p.ktile = reinterpret_cast<int4 *>(m + M.ktile);
  p.qorder = M.qorder ? reinterpret_cast<int2 *>(m + M.qorder) : nullptr;
  p.korder = M.korder ? reinterpret_cast<int2 *>(m + M.korder) : nullptr;
  if (a->cu_seqlens) {
    p.seg_q = p.seg_k = reinterpret_cast<int *>(m + M.seg);
    if (a->cu_seqlens_k) {
      p.seg_k = reinterpret_cast<int *>(m + M.segk);
      p.qoff = reinterpret_cast<int *>(m + M.qoff);
      p.koff = reinterpret_cast<int *>(m + M.koff);
    }
  } else {
    p.seg_q = a->seg_q;
    p.seg_k = a->seg_k;
  }
}

Params make_params(const attn_args *a, char *ws, const Layout &L) {
  Params p;
  memset(&p, 0, sizeof(p));
  p.B = a->B; p.Sq = a->Sq; p.Sk = a->Sk; p.Hq = a->Hq; p.Hkv = a->Hkv; p.D = a->D;
  p.G = a->Hq / a->Hkv;
  p.causal = a->causal ? 1 : 0;
  p.window = a->window > 0 ? a->window : 0;
  p.cap = a->softcap;
  p.inv_cap = a->softcap > 0.f ? 1.0f / a->softcap : 0.f;
  p.scale = a->scale;
  p.q = a->q; p.k = a->k; p.v = a->v;
  p.q_sb = a->q_stride_b; p.q_ss = a->q_stride_s; p.q_sh = a->q_stride_h;
  p.k_sb = a->k_stride_b; p.k_ss = a->k_stride_s; p.k_sh = a->k_stride_h;
  p.v_sb = a->v_stride_b; p.v_ss = a->v_stride_s; p.v_sh = a->v_stride_h;
  p.bias = a->bias;
  p.bias_sb = a->bias_stride_b; p.bias_sh = a->bias_stride_h;
  p.bias_B = a->bias_stride_b ? a->B : 1;
  p.bias_H = a->bias_stride_h ? a->Hq : 1;
  {
    const int64_t vec = a->dtype == ATTN_DTYPE_BF16 ? 8 : 4;  // elements per 16 bytes
    p.bias_vec = a->bias && a->Sk % vec == 0 && a->bias_stride_b % vec == 0 && a->bias_stride_h % vec == 0;
  }
  p.sink = a->sink;
  p.off_by_one = a->softmax_type == ATTN_SOFTMAX_OFF_BY_ONE ? 1 : 0;
  p.status = reinterpret_cast<unsigned *>(ws);
  if (needs_meta(a)) set_meta(a, a->meta ? static_cast<char *>(const_cast<void *>(a->meta)) : ws + L.meta, p);
  return p;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Pending profiling events of this host thread (attn_profile_next_main_kernel,
// attn_profile_next_aux_kernels).
thread_local cudaEvent_t t_ev_start = nullptr, t_ev_end = nullptr;
thread_local cudaEvent_t t_aux[4] = {nullptr, nullptr, nullptr, nullptr};

struct MainKernelEvents {
  cudaEvent_t start, end;
  cudaStream_t st;
  MainKernelEvents(cudaStream_t s) : start(t_ev_start), end(t_ev_end), st(s) {
    t_ev_start = t_ev_end = nullptr;
    if (start) cudaEventRecord(start, st);
  }
  void done() {
    if (end) cudaEventRecord(end, st);
    end = nullptr;
  }
};

// Builds the metadata that p points at (K1), unless the caller passed metadata built before.
int run_meta(const attn_args *a, const Params &p, cudaStream_t st, bool standalone = false) {
  if (!needs_meta(a) || (a->meta && !standalone)) return ATTN_OK;
  const MetaLayout M = meta_layout(a);
  char *m = reinterpret_cast<char *>(const_cast<unsigned char *>(p.seg_mono)) - M.mono;
  MetaOut o;
  o.clear_status = standalone ? 1 : 0;
  o.seg_q = a->cu_seqlens ? const_cast<int *>(p.seg_q) : nullptr;
  o.seg_k = a->cu_seqlens_k ? const_cast<int *>(p.seg_k) : nullptr;
  o.qoff = const_cast<int *>(p.qoff);
  o.koff = const_cast<int *>(p.koff);
  o.qrange = const_cast<int2 *>(p.qrange);
  o.krange = const_cast<int2 *>(p.krange);
  o.qrun = const_cast<int2 *>(p.qrun);
  o.krun = const_cast<int2 *>(p.krun);
  o.mono = const_cast<unsigned char *>(p.seg_mono);
  o.qtile = const_cast<int4 *>(p.qtile);
  o.ktile = const_cast<int4 *>(p.ktile);
  o.qwork = reinterpret_cast<long long *>(m + M.qwork);
  o.kwork = reinterpret_cast<long long *>(m + M.kwork);
  o.qorder = const_cast<int2 *>(p.qorder);
  o.korder = const_cast<int2 *>(p.korder);
  // The lists are only read by grids that follow them (at most four waves): when neither the
  // forward's nor the backward's grid would, the sort is left out.
  const long long fwd_blk = (long long)((a->Sq + 127) / 128) * a->Hq * a->B;
  const long long bwd_blk = (long long)((a->Sk + 127) / 128) * a->Hkv * a->B;
  if (!follow_work_list(fwd_blk) && !follow_work_list(bwd_blk)) o.qorder = o.korder = nullptr;
  return cuda_status(launch_mask_meta(p, a->cu_seqlens, a->cu_seqlens_k, a->nseq, o, st));
}

}  // namespace

int fwd_precheck(const attn_args *a, const void *O, const float *LSE, bool *empty) {
  *empty = false;
  const int s = validate(a);
  if (s != ATTN_OK) return s;
  if (a->B == 0 || a->Sq == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (!O || !LSE || !aligned16(O)) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

size_t attn_fwd_workspace_size(const attn_args *a) {
  if (validate(a) != ATTN_OK) return 0;
  return layout(a, false).total;
}

size_t attn_meta_size(const attn_args *a) {
  if (validate(a) != ATTN_OK) return 0;
  return meta_layout(a).total;
}

int attn_meta_build(const attn_args *a, void *meta, size_t meta_bytes, attn_stream_t stream) {
  const int s = validate(a);
  if (s != ATTN_OK) return s;
  const MetaLayout M = meta_layout(a);
  if (M.total == 0) return ATTN_OK;  // nothing to build
  if (!meta || meta_bytes < M.total || ((uintptr_t)meta % kAlign) != 0) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Params p;
  memset(&p, 0, sizeof(p));
  p.B = a->B; p.Sq = a->Sq; p.Sk = a->Sk;
  p.causal = a->causal ? 1 : 0;
  p.window = a->window > 0 ? a->window : 0;
  p.status = static_cast<unsigned *>(meta);  // this buffer's own status area
  set_meta(a, static_cast<char *>(meta), p);
  return run_meta(a, p, st, true);  // the metadata kernel clears the status area first
}

size_t attn_bwd_workspace_size(const attn_args *a) {
  if (validate(a) != ATTN_OK) return 0;
  return layout(a, true).total;
}

const char *attn_path_name(const attn_args *a) {
  if (validate(a) != ATTN_OK) return "";
  return use_tc(a) ? (use_tc_bwd(a) || use_wide_bwd(a) ? "tc" : "tc-fwd/simt-bwd") : "simt";
}

int attn_fwd(const attn_args *a, void *O, float *LSE, void *ws, size_t ws_bytes, attn_stream_t stream) {
  bool empty = false;
  int s = fwd_precheck(a, O, LSE, &empty);
  if (s != ATTN_OK || empty) return s;
  const Layout L = layout(a, false);
  if (!ws || ws_bytes < L.total || ((uintptr_t)ws % kAlign) != 0) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Params p = make_params(a, static_cast<char *>(ws), L);
  p.O = O;
  p.LSE = LSE;
  if (split_kv(a)) {
    p.kv_splits = a->kv_splits;
    p.o_part = reinterpret_cast<float *>(static_cast<char *>(ws) + L.o_part);
    p.lse_part = reinterpret_cast<float *>(static_cast<char *>(ws) + L.lse_part);
  }
  if ((s = run_meta(a, p, st)) != ATTN_OK) return s;
  MainKernelEvents ev(st);
  cudaError_t e = use_tc(a) ? tc_forward(p, st) : simt_forward(p, a->dtype, st);
  if (e == cudaSuccess && p.kv_splits > 1) e = launch_splitkv_merge(p, st);
  ev.done();
  return cuda_status(e);
}

int attn_bwd(const attn_args *a, const void *O, const float *LSE, const void *dO, void *dQ, void *dK,
             void *dV, void *dbias, float *dsink, void *ws, size_t ws_bytes, attn_stream_t stream) {
  int s = validate(a);
  if (s != ATTN_OK) return s;
  if (a->B > 0 && a->Sq > 0 && (!O || !LSE || !dO || !dQ)) return ATTN_ERR_INVALID;
  if (a->B > 0 && a->Sk > 0 && (!dK || !dV)) return ATTN_ERR_INVALID;
  if (!aligned16(O) || !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
    return ATTN_ERR_INVALID;
  if ((a->bias != nullptr) != (dbias != nullptr)) return ATTN_ERR_INVALID;
  if ((a->sink != nullptr) != (dsink != nullptr)) return ATTN_ERR_INVALID;
  if (a->B == 0) return ATTN_OK;
  const Layout L = layout(a, true);
  if (!ws || ws_bytes < L.total || ((uintptr_t)ws % kAlign) != 0) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t esz = a->dtype == ATTN_DTYPE_BF16 ? 2 : 4;
  if (a->Sq == 0) {  // no query rows: every gradient is zero
    const size_t kv = (size_t)a->B * a->Sk * a->Hkv * a->D * esz;
    if (cudaMemsetAsync(dK, 0, kv, st) != cudaSuccess || cudaMemsetAsync(dV, 0, kv, st) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (dsink && cudaMemsetAsync(dsink, 0, a->Hq * sizeof(float), st) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  char *w = static_cast<char *>(ws);
  Params p = make_params(a, w, L);
  p.O = const_cast<void *>(O);
  p.LSE = const_cast<float *>(LSE);
  p.dO = dO;
  p.dQ = dQ; p.dK = dK; p.dV = dV; p.dbias = dbias; p.dsink = dsink;
  p.Dvec = reinterpret_cast<float *>(w + L.dvec);
  p.sq_pad = (a->Sq + 127) / 128 * 128;
  p.dsink_part = a->sink ? reinterpret_cast<float *>(w + L.dsink_part) : nullptr;
  p.n_part = bwd_pre_partials(a->B, a->Sq, a->Hq);
  const bool tc = use_tc_bwd(a), wide = !tc && use_wide_bwd(a);
  p.dQacc = tc ? reinterpret_cast<float *>(w + L.dqacc) : nullptr;
  p.lse2p = tc || wide ? reinterpret_cast<float *>(w + L.lse2) : nullptr;
  p.dsplit = tc && tc_bwd_fused(a->D) ? reinterpret_cast<uint4 *>(w + L.dsplit) : nullptr;
  p.dbias_acc = a->bias ? reinterpret_cast<float *>(w + L.dbias_acc) : nullptr;
  // Group-major backward grid for long query ranges without segments (see bwd_tc.cu).
  p.bwd_group_major = (!needs_meta(a) && (a->window > 0 ? std::min(a->window, a->Sq) : a->Sq) >= 16384) ? 1 : 0;
  if ((s = run_meta(a, p, st)) != ATTN_OK) return s;
  if (a->bias && cudaMemsetAsync(p.dbias_acc, 0, dbias_elems(a) * sizeof(float), st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  cudaEvent_t aux[4];
  for (int x = 0; x < 4; ++x) {
    aux[x] = t_aux[x];
    t_aux[x] = nullptr;
  }
  if (aux[0]) cudaEventRecord(aux[0], st);
  if ((s = cuda_status(launch_bwd_pre(p, a->dtype, tc, st))) != ATTN_OK) return s;
  if (aux[1]) cudaEventRecord(aux[1], st);
  {
    MainKernelEvents ev(st);
    cudaError_t e = tc ? tc_backward(p, st) : wide ? wide_backward(p, w + L.wide, st) : simt_backward(p, a->dtype, st);
    ev.done();
    if ((s = cuda_status(e)) != ATTN_OK) return s;
  }
  if (aux[2]) cudaEventRecord(aux[2], st);
  s = cuda_status(launch_bwd_post(p, a->dtype, tc, dbias_elems(a), st));
  if (aux[3]) cudaEventRecord(aux[3], st);
  return s;
}

int attn_check_device_status(void *ws, attn_stream_t stream) {
  if (!ws) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word == 0) return ATTN_OK;
  if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return ATTN_ERR_CUDA;  // detail words stay
  return ATTN_ERR_DEVICE;
}

void attn_profile_next_main_kernel(void *ev_start, void *ev_end) {
  t_ev_start = static_cast<cudaEvent_t>(ev_start);
  t_ev_end = static_cast<cudaEvent_t>(ev_end);
}

void attn_profile_next_aux_kernels(void *pre_start, void *pre_end, void *post_start, void *post_end) {
  t_aux[0] = static_cast<cudaEvent_t>(pre_start);
  t_aux[1] = static_cast<cudaEvent_t>(pre_end);
  t_aux[2] = static_cast<cudaEvent_t>(post_start);
  t_aux[3] = static_cast<cudaEvent_t>(post_end);
}

uint64_t attn_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

const char *attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE: return "device-side error recorded by a kernel";
    default: return "unknown status";
  }
}

}  // extern "C"
