/*
 * attn_gb300.h -- C ABI of the GB300 (sm_103a) fused attention library.
 *
 * One fused attention forward and backward with these score modifications:
 *   - tanh logit soft-capping t = cap * tanh(u / cap), applied after the scale and the
 *     additive bias and before masking; its backward chains 1 - tanh^2(u / cap) into dS,
 *     taken from the finite pre-mask logit
 *       (TransformerEngine PR #3391 "Thread tanh logit softcapping through FlashAttention",
 *        intro and "What changed"; openxla/tokamax PR #1121 "Support logits soft-capping in
 *        the Pallas-Triton attention VJP", PR body);
 *   - a learnable attention sink: one extra softmax column of logit sink[h] per query head,
 *     entering each row exactly once and carrying no value; its gradient is
 *     dsink[h] = -sum_{b,i} p_sink(b,h,i) * (dO_i . O_i)
 *       (TransformerEngine PR #3551, "What was broken" / "What changed");
 *   - the off-by-one softmax: the same extra column with its logit fixed at 0 for every
 *     head and no gradient (the "off-by-one" softmax type that TransformerEngine PR #3551
 *     tests beside "learnable", "Verification" table; the page gives no formula -- this is
 *     the learnable sink at its default zero offset, held fixed);
 *   - GQA/MQA: query head h reads kv head h / (Hq / Hkv);
 *   - causal, sliding-window and packed-segment masks (segment ids or cu_seqlens)
 *       (MaxText commit message quoted on tokamax PR #1121: sliding window, packing with
 *        segment ids lowered to cu_seqlens);
 *   - an optional post-scale additive bias ("post_scale_bias", TransformerEngine PR #3551,
 *     Greptile finding "Offset Corrupts Bias Gradient Shape": dbias takes the bias's shape).
 *
 * Definition (per batch b, query head h, kv head g = h / (Hq / Hkv), query i, key j):
 *   u_ij   = scale * q_i . k_j + bias[b,h,i,j]
 *   t_ij   = softcap > 0 ? softcap * tanh(u_ij / softcap) : u_ij
 *   vis_ij = (!causal || j <= i + Sk - Sq) && (window <= 0 || (i + Sk - Sq) - j < window)
 *            && (no segments || seg_q[b,i] == seg_k[b,j])
 *   LSE_i  = ln( [sink ? exp(sink[h]) : off-by-one ? 1 : 0] + sum_{vis} exp(t_ij) )
 *                                                                         (natural log)
 *   O_i    = sum_{vis} exp(t_ij - LSE_i) v_j
 * A row with nothing visible gets O = 0 and zero gradients, with LSE = -inf -- or, with a
 * sink or the off-by-one column, LSE = that column's logit.
 *
 * Layout: "bshd".  q, O, dO, dQ are [B, Sq, Hq, D]; k, v, dK, dV are [B, Sk, Hkv, D].
 * q, k, v may be strided (element strides for b, s, h; d is contiguous); O, dO, dQ, dK, dV
 * are dense.  LSE is float [B, Hq, Sq].  All device pointers.
 *
 * Ownership: the caller allocates every input, output and workspace; the library allocates
 * no device memory and keeps no state besides one-time kernel attributes (set on first use
 * per device; thread-safe).  Every call is asynchronous on `stream` and never synchronises,
 * except attn_check_device_status.  Calls on distinct streams with distinct workspaces may
 * run concurrently.
 *
 * Errors: every call validates its arguments first.  On any synchronous error no kernel is
 * launched and no output is written.  Kernels that give up a bounded wait record it in the
 * workspace's status word (read with attn_check_device_status) and exit cleanly; they never
 * trap or spin forever.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *attn_stream_t;

enum attn_dtype {
    ATTN_DTYPE_BF16 = 1,  /* q, k, v, bias, O, dO, dQ, dK, dV, dbias in bfloat16       */
    ATTN_DTYPE_F32 = 2    /* ... in float32 (fp32 FFMA kernels, for tight tolerances)   */
};

enum attn_softmax_type {
    ATTN_SOFTMAX_DEFAULT = 0,     /* plain softmax, or the learnable sink when sink != NULL */
    ATTN_SOFTMAX_OFF_BY_ONE = 1   /* one extra column of logit 0 per row; sink must be NULL,
                                     and there is no dsink                                   */
};

enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,      /* null required pointer, bad shape/stride/alignment,
                                  negative or NaN softcap, non-finite scale, ...          */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not built: D > 512; cu_seqlens together with
                                  seg_q / seg_k                                          */
    ATTN_ERR_WORKSPACE = 3,    /* ws NULL or smaller than the size query returned        */
    ATTN_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed            */
    ATTN_ERR_DEVICE = 5        /* a kernel recorded a device-side error (bounded wait
                                  expired, malformed cu_seqlens) -- attn_check_device_status */
};

typedef struct {
    int dtype;                 /* enum attn_dtype                                          */
    int B, Sq, Sk, Hq, Hkv, D; /* B, Sq, Sk >= 0 (B == 0 or Sq == 0: nothing to compute);
                                  Hq, Hkv >= 1 with Hq % Hkv == 0; D % 8 == 0, D <= 512.
                                  Tensor-core kernels: bf16 with Sk > 0 and D in {64, 128,
                                  256}, or D in {320, 384, 448, 512} (the wide form for
                                  MaxText's chunked head-dim accumulation above 256, tokamax
                                  PR #1121: two CTAs per query tile, each producing part of
                                  O; its backward is a scores kernel and three GEMMs through
                                  two bf16 scratch planes of B*Hq*Sq_pad*Sk_pad elements
                                  (Sq, Sk rounded up to 128) in the workspace, taken while
                                  they stay within 16 GiB), with or without a bias, sink,
                                  segments or splits.  The fp32 FFMA kernels take every
                                  other call: fp32 inputs, other head dims, and wide-form
                                  backwards whose planes would exceed 16 GiB.              */
    const void *q;             /* [B,Sq,Hq,D] with the strides below (elements)           */
    int64_t q_stride_b, q_stride_s, q_stride_h;
    const void *k;             /* [B,Sk,Hkv,D]                                             */
    int64_t k_stride_b, k_stride_s, k_stride_h;
    const void *v;             /* [B,Sk,Hkv,D]                                             */
    int64_t v_stride_b, v_stride_s, v_stride_h;
    /* Optional additive bias, logically [B,Hq,Sq,Sk]: element (b,h,i,j) lives at
     * bias[b*bias_stride_b + h*bias_stride_h + i*Sk + j]; a stride of 0 broadcasts that
     * dimension.  NULL: no bias.  Same dtype as q; 16-byte aligned base.  Added after the
     * scale and before the cap.  Rows that start on 16-byte boundaries (Sk and both strides
     * multiples of 8 bf16 elements) are read with 16-byte loads, others element by element. */
    const void *bias;
    int64_t bias_stride_b, bias_stride_h;
    /* Optional packed segments: seg_q [B,Sq] and seg_k [B,Sk] int32 (both or neither; the
     * same array for both when Sq == Sk).  A pair is visible only if the ids are equal.  Any
     * ids are accepted; runs of non-decreasing ids additionally let the kernels skip whole
     * tiles.  With Sq != Sk, causal and window keep the one bottom-right alignment below (ids
     * carry no per-sequence offsets; cu_seqlens_k gives those).                            */
    const int32_t *seg_q, *seg_k;
    /* Alternative to seg_q/seg_k (not both): cu_seqlens [nseq+1] int32 with
     * cu_seqlens[0] == 0, non-decreasing, cu_seqlens[nseq] <= Sq; requires B == 1 and, unless
     * cu_seqlens_k gives the keys their own boundaries, Sq == Sk.  Token t belongs to sequence s with cu[s] <= t < cu[s+1]; tokens at or past
     * cu[nseq] form one extra trailing sequence.  A malformed array is reported through the
     * device status word.                                                                  */
    const int32_t *cu_seqlens;
    int nseq;
    int causal;                /* nonzero: key j visible to query i only if j <= i + Sk - Sq */
    int window;                /* > 0: key j visible only if (i + Sk - Sq) - j < window      */
    float softcap;             /* 0: off; > 0: cap; negative, NaN or inf: ATTN_ERR_INVALID  */
    const float *sink;         /* optional [Hq] float sink logits; NULL: no sink            */
    float scale;               /* finite; usually 1/sqrt(D)                                 */
    int softmax_type;          /* enum attn_softmax_type; zero-initialised = DEFAULT.  Any
                                  other value, or OFF_BY_ONE with a sink: ATTN_ERR_INVALID  */
    /* Split-KV forward, for rows too few to fill the GPU (decode-like shapes, long keys):
     * 0 or 1: off.  n in 2..64: the tensor-core forward splits every query tile's visible key
     * tiles into n contiguous shares, one CTA each, and a merge kernel combines their
     * normalised partial outputs and log-normalisers, adding the sink or off-by-one column
     * exactly once per row (TransformerEngine PR #3551, "What changed": the sink enters each
     * row once when tiles' statistics are merged).  The workspace grows by
     * n * B * Hq * Sq * (D + 1) * 4 bytes.  Results equal the unsplit forward up to rounding.
     * Head dims above 256 and the FFMA path (fp32 inputs, other head dims) compute unsplit.  Other
     * values: ATTN_ERR_INVALID.  The backward ignores this field.                           */
    int kv_splits;
    /* Optional key boundaries for cu_seqlens ("thd" varlen with Sq != Sk per sequence):
     * cu_seqlens_k [nseq+1] int32 with the same rules on the key axis (cu_seqlens_k[nseq] <=
     * Sk).  Sequence s then holds queries [cu_seqlens[s], cu_seqlens[s+1]) and keys
     * [cu_seqlens_k[s], cu_seqlens_k[s+1]); tokens past either end form the trailing sequence
     * nseq.  Causal and window masks align bottom-right within every sequence: with
     * off_s = end_k(s) - end_q(s), key j is visible to query i of the same sequence iff
     * (!causal || j <= i + off_s) && (window <= 0 || i + off_s - j < window), so a sequence
     * with more queries than keys has leading queries that see nothing (MaxText commit message
     * quoted on tokamax PR #1121: packing lowered to per-segment q / kv seqlens and offsets).
     * Requires cu_seqlens; Sq == Sk is then not required.  NULL: the keys share cu_seqlens.  */
    const int32_t *cu_seqlens_k;
    /* Optional mask metadata built by attn_meta_build for these same arguments (same shapes,
     * masks and segment / cu_seqlens arrays -- the library cannot check this), 256-byte
     * aligned.  With segments or cu_seqlens, attn_fwd and attn_bwd then read it instead of
     * building it in their workspaces (whose size query shrinks accordingly): build it once per
     * step and pass it to both.  NULL: each call builds its own.  Ignored without segments.  */
    const void *meta;
} attn_args;

/*
 * Mask metadata (segment ids or cu_seqlens; MaxText commit message quoted on tokamax PR #1121:
 * packing with segment ids lowered to per-segment boundaries, run starts per row, boundaries
 * not aligned to tiles).  For each batch row: the effective segment ids (from cu_seqlens), the
 * per-token bottom-right offsets (cu_seqlens_k), whether the ids are sorted, the key range of
 * every 64-row query tile and the query range of every 64-key tile; for every 128-row query
 * tile and 128-key tile its class bounds (the keys some row sees, the keys every row sees:
 * FULL / PARTIAL / EMPTY key tiles) and its visible pairs; and, with at most 4096 tiles per
 * axis, the longest-first work lists (tiles in descending order of visible pairs) that the
 * tensor-core grids follow.
 *
 * attn_meta_size: bytes of the metadata buffer (256-byte multiple), or 0 when the arguments
 * need none (no segments / cu_seqlens, B == 0) or are invalid.
 * attn_meta_build: builds it into `meta` (256-byte aligned, at least attn_meta_size bytes),
 * asynchronously on `stream`; pass the buffer as args->meta to attn_fwd and attn_bwd.  The
 * buffer's first 256 bytes are its own status area, cleared by each build: a malformed
 * cu_seqlens / cu_seqlens_k is recorded there (read with attn_check_device_status(meta,
 * stream)).  Returns an attn_status; ATTN_OK without launching when nothing is needed.
 */
size_t attn_meta_size(const attn_args *a);
int attn_meta_build(const attn_args *a, void *meta, size_t meta_bytes, attn_stream_t stream);

/* Bytes of workspace attn_fwd needs for these arguments (256-byte multiple, >= 256). */
size_t attn_fwd_workspace_size(const attn_args *a);

/*
 * Forward: O [B,Sq,Hq,D] (dtype of q) and LSE [B,Hq,Sq] float (natural log, sink included).
 * ws: device workspace of at least attn_fwd_workspace_size(a) bytes, 256-byte aligned,
 * zero-filled once before its first use (its first 256 bytes hold the sticky device status
 * word).  Returns an attn_status.
 */
int attn_fwd(const attn_args *a, void *O, float *LSE, void *ws, size_t ws_bytes,
             attn_stream_t stream);

/*
 * attn_fwd without a caller-provided workspace, for callers that cannot allocate device
 * memory: plugins hosted by a runtime that owns every device allocation and hands them no
 * allocator, or deployments whose device-memory budget is fixed up front.  The pages this
 * library follows have no counterpart to this entry point.
 *
 * Computes exactly what attn_fwd computes (same arguments, same outputs), with its scratch
 * taken from a 4 MiB array compiled into the library (one per GPU context that loads the
 * library, resident until the process exits).  It makes attn_fwd's checks in attn_fwd's
 * order and answers them alike (B == 0 or Sq == 0: ATTN_OK, nothing launched); a request that
 * passes them but whose attn_fwd_workspace_size exceeds 4 MiB is then rejected with
 * ATTN_ERR_WORKSPACE before anything is launched.  It allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Every call looks up the array's device address in the context that is current (the first
 * call in a context loads the library's device code there); make the first call on a device
 * before any stream capture.  Every call shares the array: calls whose work overlaps on the
 * GPU (other streams, other threads) race and must not be issued.  Each call clears the
 * array's status word at its start; attn_noalloc_check_device_status reads what the most
 * recent call recorded there.
 */
int attn_fwd_noalloc(const attn_args *a, void *O, float *LSE, attn_stream_t stream);

/*
 * attn_check_device_status for attn_fwd_noalloc: synchronises `stream`, reads and clears the
 * status word of the built-in array in the current context.  Returns ATTN_OK, ATTN_ERR_DEVICE
 * (the most recent attn_fwd_noalloc call on this device recorded a device-side error: an
 * expired bounded wait, or a malformed cu_seqlens / cu_seqlens_k) or ATTN_ERR_CUDA.  Like the
 * entry point itself, it allocates nothing and has no counterpart on the pages.
 */
int attn_noalloc_check_device_status(attn_stream_t stream);

/* Bytes of workspace attn_bwd needs (same rules as attn_fwd_workspace_size). */
size_t attn_bwd_workspace_size(const attn_args *a);

/*
 * Backward of O with respect to q, k, v, bias and sink, given dO.
 *   O, LSE: the forward's outputs for the same arguments; dO [B,Sq,Hq,D] dense.
 *   dQ [B,Sq,Hq,D], dK/dV [B,Sk,Hkv,D]: dense outputs, overwritten.
 *   dbias: required iff a->bias != NULL; dense with the bias's own shape
 *          [bias_stride_b ? B : 1, bias_stride_h ? Hq : 1, Sq, Sk]; broadcast dimensions are
 *          summed over; overwritten.
 *   dsink: required iff a->sink != NULL; float [Hq], summed over every batch and row;
 *          overwritten (not accumulated).
 * The 1 - tanh^2(u/cap) factor is applied before dK, dQ and dbias are formed, so those are
 * gradients with respect to the pre-cap logits (tokamax PR #1121, PR body).
 */
int attn_bwd(const attn_args *a, const void *O, const float *LSE, const void *dO,
             void *dQ, void *dK, void *dV, void *dbias, float *dsink,
             void *ws, size_t ws_bytes, attn_stream_t stream);

/*
 * Synchronises `stream`, reads and clears the workspace's device status word.
 * Returns ATTN_OK, ATTN_ERR_DEVICE (a kernel recorded an error since the last check) or
 * ATTN_ERR_CUDA (the stream itself reported an error).
 */
int attn_check_device_status(void *ws, attn_stream_t stream);

/*
 * Self-test of the bounded-wait failure path (TransformerEngine PR #3391, "What changed":
 * fail closed, never return a silently wrong result).  Launches one small kernel on `stream`
 * whose first wait is on an mbarrier that nothing completes, with limit_ns as its time limit
 * (1 us .. 2 s); the kernels' own waits behind it give up on the status bit.  Afterwards the
 * workspace holds exactly what a real expired wait leaves: attn_check_device_status(ws)
 * returns ATTN_ERR_DEVICE; status words 1..6 hold 1, the barrier's shared-memory address and
 * parity (0), the CTA (0) and the thread (0) of the first wait to give up; words 10 and 11 the
 * barrier and parity | 0x100 of warp 1 of that CTA; words 48 and 49 the addresses of the two
 * barriers, for comparison.  Until that status is read and cleared, attn_fwd / attn_bwd with
 * this workspace return from their kernels at once.  ws: at least 256 bytes, 256-byte
 * aligned, zero-filled.  Nothing faults or traps; the context stays usable.
 */
int attn_selftest_wait_expiry(void *ws, size_t ws_bytes, uint64_t limit_ns, attn_stream_t stream);

/* Static description of a status code (never NULL). */
const char *attn_status_string(int status);

/* Kernel path the forward / backward would take for these arguments, for tests and
 * profiling: "tc" (tcgen05 tensor-core kernels), "simt" (FFMA kernels), or "" when the
 * arguments are rejected.  Static string. */
const char *attn_path_name(const attn_args *a);

/*
 * Profiling hook: the next attn_fwd or attn_bwd call made by this host thread records
 * `ev_start` (a cudaEvent_t) on its stream immediately before launching its main kernel
 * (the tensor-core or FFMA attention kernel; for the FFMA backward, the first of its two)
 * and `ev_end` immediately after its last main kernel (with kv_splits, the merge), then
 * forgets both.  Passing NULLs
 * cancels a pending request.  Adds no work to the call.
 */
void attn_profile_next_main_kernel(void *ev_start, void *ev_end);

/*
 * Profiling hook for the memory-bound kernels of the next attn_bwd call made by this host
 * thread: it records `pre_start` / `pre_end` (cudaEvent_t) on its stream immediately before
 * and after the preprocess kernel (D = rowsum(dO * O), LSE * log2(e), the sink gradient's
 * partial sums, the fp32 dQ accumulator zeroed) and `post_start` / `post_end` around the
 * postprocess kernel (dQ converted, dsink and dbias written out), then forgets all four.
 * NULLs cancel a pending request.  Adds no work to the call.
 */
void attn_profile_next_aux_kernels(void *pre_start, void *pre_end, void *post_start, void *post_end);

/* Number of kernels this library has launched in this process (all devices), for
 * accounting in benchmarks; monotonic, thread-safe. */
uint64_t attn_launch_counter(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
