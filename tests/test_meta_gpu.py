"""The mask metadata kernel (K1) on the GPU: per-token visible intervals, tile classes, per-tile
work and the longest-first work lists, checked against the oracle's visibility (the mask definition, pair by pair), and
the metadata built once and shared by attn_fwd and attn_bwd (MaxText commit message quoted on
tokamax PR #1121: packed rows, run starts per row, boundaries not aligned to tiles)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity import (TOL, compare_full, frob_rel, full_oracle, problem_from_inputs, run_gpu, to64,
                    varlen_oracle)
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _up(x):
    return (x + 255) // 256 * 256


def meta_regions(B, Sq, Sk, cu=False, cuk=False):
    """Byte offsets of the metadata buffer's regions, in the order the library lays them out
    (mirrored here to read the buffer back; the total is checked against attn_meta_size)."""
    nq, nk = -(-Sq // 64), -(-Sk // 64)
    nq128, nk128 = -(-Sq // 128), -(-Sk // 128)
    r, off = {}, 256
    for name, size in [("mono", B), ("qrange", B * nq * 8), ("krange", B * nk * 8), ("qrun", B * Sq * 8),
                       ("krun", B * Sk * 8)]:
        r[name], off = off, off + _up(size)
    if cu:
        r["seg"], off = off, off + _up(Sq * 4)
    if cuk:
        for name, size in [("segk", Sk * 4), ("qoff", Sq * 4), ("koff", Sk * 4)]:
            r[name], off = off, off + _up(size)
    for name, size in [("qtile", B * nq128 * 16), ("ktile", B * nk128 * 16), ("qwork", B * nq128 * 8),
                       ("kwork", B * nk128 * 8), ("qorder", B * nq128 * 8), ("korder", B * nk128 * 8)]:
        r[name], off = off, off + _up(size)
    r["total"] = off
    return r


def _read(buf, off, n, dtype, width=1):
    a = buf[off:off + n * width * np.dtype(dtype).itemsize].view(dtype)
    return a.reshape(n, width) if width > 1 else a


def _check_runs(runs, count, first, last, sorted_ids):
    """Per-token intervals [B*n_rows, 2] against the oracle's per-row counts / first / last: with
    sorted ids exactly the visible run; with unsorted ids an interval holding every visible
    pair (the kernels then test ids pair by pair)."""
    runs = runs.reshape(count.shape + (2,))
    seen = count > 0
    lo, hi = runs[..., 0], runs[..., 1]
    assert np.all(lo[seen] <= first[seen]) and np.all(hi[seen] >= last[seen] + 1)
    if sorted_ids:
        assert np.array_equal(lo[seen], first[seen]) and np.array_equal(hi[seen], last[seen] + 1)
        assert np.all(lo[~seen] >= hi[~seen])


def _check_axis(tiles, work, order, count, first, last, n_other, sorted_ids, B, n_rows, key_axis):
    """tiles [B*nt, 4] {lo, hi, flo, fhi}, work [B*nt], order [B*nt, 2] against the oracle's
    per-row visible counts / first / last ([B, n_rows])."""
    nt = -(-n_rows // 128)
    works = []
    for b in range(B):
        for t in range(nt):
            rows = slice(t * 128, min(t * 128 + 128, n_rows))
            c, f, l = count[b, rows], first[b, rows], last[b, rows]
            lo, hi, flo, fhi = tiles[b * nt + t]
            w = int(work[b * nt + t])
            if sorted_ids:
                assert w == int(c.sum()), (b, t, w, int(c.sum()))
            else:
                assert w >= int(c.sum())  # an upper bound: the kernels test pairs one by one
            seen = c > 0
            if seen.any():  # union of the rows' visible sets (EMPTY outside it)
                assert lo <= f[seen].min() and hi >= l[seen].max() + 1, (b, t)
                if sorted_ids:
                    assert (lo, hi) == (f[seen].min(), l[seen].max() + 1), (b, t)
            else:
                assert lo >= hi
            if flo < fhi:  # FULL keys: every row sees every one of them
                assert sorted_ids and seen.all()
                assert not key_axis or (t + 1) * 128 <= n_rows  # no FULL steps in a ragged key tile
                assert np.all(f <= flo) and np.all(l >= fhi - 1), (b, t)
                assert np.all(c >= l - f + 1)  # sorted runs: each row's visible set is an interval
            works.append(w)
    works = np.array(works)
    # the work list: every tile once, in descending power-of-two class of its visible pairs,
    # and within a class in the grid's locality order (query tiles latest first, key tiles
    # earliest first, batch row fastest)
    idx = order[:, 0] * nt + order[:, 1]
    assert sorted(idx.tolist()) == list(range(B * nt))
    cls = np.array([int(w + 1).bit_length() for w in works[idx]])
    assert np.all(np.diff(cls) <= 0)
    t = order[:, 1] if key_axis else nt - 1 - order[:, 1]
    rank = t * B + order[:, 0]
    for e in range(len(idx) - 1):
        if cls[e] == cls[e + 1]:
            assert rank[e] < rank[e + 1]


CASES = [
    # packed rows: runs ~ U[40, 400], boundaries not on tile multiples; causal
    (Workload("meta_packed", "bf16", B=2, Sq=1000, Sk=1000, Hq=2, Hkv=1, D=64, causal=True, segments=True,
              run_lo=40, run_hi=400), None),
    # packed, non-causal, with a window
    (Workload("meta_packed_window", "bf16", B=3, Sq=700, Sk=700, Hq=2, Hkv=1, D=64, causal=False, window=90,
              segments=True, run_lo=20, run_hi=300), None),
    # interleaved (unsorted) ids: no FULL tiles, work an upper bound
    (Workload("meta_interleaved", "bf16", B=1, Sq=500, Sk=500, Hq=2, Hkv=1, D=64, causal=True), "interleaved"),
]


@pytest.mark.parametrize("w,kind", CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_tile_classes_work_and_order_against_the_oracle(w, kind):
    import attention_flash_attn_gb300 as fa
    inp = make_inputs(w)
    seg = inp["seg"] if kind is None else (torch.arange(w.Sq, dtype=torch.int32) % 3).view(1, -1).repeat(w.B, 1)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    meta = fa.attn_meta(t["q"], t["k"], t["v"], causal=w.causal, window=w.window, seg_q=seg.cuda())
    torch.cuda.synchronize()
    r = meta_regions(w.B, w.Sq, w.Sk)
    assert meta.numel() == r["total"]
    buf = meta.cpu().numpy()
    sorted_ids = bool(np.all(np.diff(seg.numpy(), axis=1) >= 0))
    assert np.array_equal(buf[r["mono"]:r["mono"] + w.B], np.full(w.B, int(sorted_ids), np.uint8))
    p = oracle.Problem(np.zeros((w.B, w.Sq, 1, 1)), np.zeros((w.B, w.Sk, 1, 1)), np.zeros((w.B, w.Sk, 1, 1)),
                       scale=1.0, causal=w.causal, window=w.window, seg_q=seg.numpy())
    nq, nk = w.B * -(-w.Sq // 128), w.B * -(-w.Sk // 128)
    _check_axis(_read(buf, r["qtile"], nq, np.int32, 4), _read(buf, r["qwork"], nq, np.int64),
                _read(buf, r["qorder"], nq, np.int32, 2), *oracle.row_visible(p), w.Sk, sorted_ids, w.B, w.Sq, False)
    _check_axis(_read(buf, r["ktile"], nk, np.int32, 4), _read(buf, r["kwork"], nk, np.int64),
                _read(buf, r["korder"], nk, np.int32, 2), *oracle.col_visible(p), w.Sq, sorted_ids, w.B, w.Sk, True)
    _check_runs(_read(buf, r["qrun"], w.B * w.Sq, np.int32, 2), *oracle.row_visible(p), sorted_ids)
    _check_runs(_read(buf, r["krun"], w.B * w.Sk, np.int32, 2), *oracle.col_visible(p), sorted_ids)


def _same_results(a, b):
    for key in ("O", "LSE", "dk", "dv", "dsink"):
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
    assert frob_rel(to64(a["dq"]), to64(b["dq"])) < 1e-6  # dQ's reduce-adds land in a run-dependent order


def test_metadata_built_once_and_shared():
    """attn_meta once, passed to attn_fwd and attn_bwd: the same results as each call building
    its own, and both against the oracle; the workspaces shrink by the metadata's size."""
    import ctypes
    import attention_flash_attn_gb300 as fa
    w = Workload("meta_shared", "bf16", B=2, Sq=1000, Sk=1000, Hq=4, Hkv=2, D=128, causal=True, softcap=30.0,
                 sink=True, segments=True, run_lo=40, run_hi=400, q_std=3.0)
    inp = make_inputs(w)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    meta = fa.attn_meta(t["q"], t["k"], t["v"], causal=w.causal, window=w.window, seg_q=t["seg"])
    own = run_gpu(w, inp)
    shared = run_gpu(w, inp, meta=meta)
    _same_results(own, shared)
    errs = compare_full(w, shared, full_oracle(w, inp))
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
    a, keep = fa.build_args(t["q"], t["k"], t["v"], causal=True, seg_q=t["seg"])
    a2, keep2 = fa.build_args(t["q"], t["k"], t["v"], causal=True, seg_q=t["seg"], meta=meta)
    L = fa.lib()
    for f in (L.attn_fwd_workspace_size, L.attn_bwd_workspace_size):
        assert f(ctypes.byref(a)) - f(ctypes.byref(a2)) == L.attn_meta_size(ctypes.byref(a)) == meta.numel()


def test_metadata_shared_with_separate_key_boundaries():
    """thd varlen (cu_seqlens + cu_seqlens_k): metadata built once, the same results, and the
    per-sequence oracle; a malformed cu_seqlens is reported in the buffer's own status word."""
    import attention_flash_attn_gb300 as fa
    w = Workload("meta_varlen", "bf16", B=1, Sq=578, Sk=1424, Hq=4, Hkv=2, D=128, causal=True, softcap=30.0,
                 sink=True, q_std=3.0)
    cu_q, cu_k = [0, 50, 180, 181, 481], [0, 200, 330, 394, 684]
    inp = make_inputs(w)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    meta = fa.attn_meta(t["q"], t["k"], t["v"], causal=True, cu_seqlens=cq, cu_seqlens_k=ck)
    own = run_gpu(w, inp, cu_seqlens=cq, cu_seqlens_k=ck)
    shared = run_gpu(w, inp, cu_seqlens=cq, cu_seqlens_k=ck, meta=meta)
    _same_results(own, shared)
    errs = compare_full(w, shared, varlen_oracle(w, inp, cu_q, cu_k))
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
    st = torch.cuda.current_stream().cuda_stream
    assert fa.lib().attn_check_device_status(meta.data_ptr(), st) == 0
    bad = torch.tensor([0, 180, 50, 181, 481], dtype=torch.int32, device="cuda")
    meta_bad = fa.attn_meta(t["q"], t["k"], t["v"], causal=True, cu_seqlens=bad, cu_seqlens_k=ck, out=meta)
    assert fa.lib().attn_check_device_status(meta_bad.data_ptr(), st) == 5


# Segment ids given per axis (seg_q [B, Sq], seg_k [B, Sk]) with Sq != Sk, one axis longer than
# the metadata kernel keeps in shared memory (49152 ids) and the other not: only the blocks of
# the long axis's tiles stage the other (short) axis's ids there.
PER_AXIS = [
    # a chunk of 200 queries continuing the last two sequences of a packed 50 000-key row (causal,
    # bottom-right): 72 queries of sequence 1, 128 of sequence 2
    (Workload("seg_per_axis_long_keys", "bf16", B=1, Sq=200, Sk=50000, Hq=2, Hkv=1, D=64, causal=True,
              softcap=30.0, sink=True, q_std=2.0), [1] * 72 + [2] * 128, [0] * 20000 + [1] * 29872 + [2] * 128),
    # 50 000 queries over 300 keys in two sequences (non-causal)
    (Workload("seg_per_axis_long_queries", "bf16", B=1, Sq=50000, Sk=300, Hq=2, Hkv=1, D=64, causal=False,
              softcap=30.0, q_std=2.0), [0] * 49800 + [1] * 200, [0] * 100 + [1] * 200),
]


@pytest.mark.parametrize("w,ids_q,ids_k", PER_AXIS, ids=lambda x: x.name if hasattr(x, "name") else None)
def test_segment_ids_per_axis_with_one_long_axis(w, ids_q, ids_k):
    """Per-token intervals against the oracle's visibility, and the forward and backward against
    the oracle, with distinct query and key ids and Sq != Sk."""
    import attention_flash_attn_gb300 as fa
    inp = {**make_inputs(w), "seg": None}
    seg_q = torch.tensor(ids_q, dtype=torch.int32).view(1, -1)
    seg_k = torch.tensor(ids_k, dtype=torch.int32).view(1, -1)
    p = dataclasses.replace(problem_from_inputs(w, inp), seg_q=seg_q.numpy(), seg_k=seg_k.numpy())
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    meta = fa.attn_meta(t["q"], t["k"], t["v"], causal=w.causal, seg_q=seg_q.cuda(), seg_k=seg_k.cuda())
    torch.cuda.synchronize()
    r = meta_regions(w.B, w.Sq, w.Sk)
    buf = meta.cpu().numpy()
    assert buf[r["mono"]] == 1
    _check_runs(_read(buf, r["qrun"], w.B * w.Sq, np.int32, 2), *oracle.row_visible(p), True)
    _check_runs(_read(buf, r["krun"], w.B * w.Sk, np.int32, 2), *oracle.col_visible(p), True)
    gpu = run_gpu(w, inp, seg_q=seg_q.cuda(), seg_k=seg_k.cuda())
    O, LSE = oracle.forward(p)
    ref = oracle.backward(p, to64(inp["dO"]), O, LSE)
    ref["O"], ref["LSE"] = O, LSE
    errs = compare_full(w, gpu, ref)
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
