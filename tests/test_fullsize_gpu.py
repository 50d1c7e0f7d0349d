"""Full-size workloads, in the launch configuration bench.py times, checked against the fp64
oracle on samples it can compute: every row of O / LSE and sampled rows of dQ and columns
of dK / dV for one (batch, kv group), plus dsink over every batch for that group.
Same tolerance as the small cases (Frobenius-relative 1e-2 for bf16)."""
import numpy as np
import pytest

import oracle
from parity import TOL, frob_rel, problem_from_inputs, run_gpu, to64
from workloads import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_positions(S, seg_row=None):
    pos = {0, 1, 63, 64, 127, 128, 129, S // 2 - 1, S // 2, S - 129, S - 128, S - 2, S - 1}
    if seg_row is not None:
        b = np.flatnonzero(np.diff(seg_row)) + 1
        for x in b[:6]:
            pos |= {int(x) - 1, int(x)}
    return sorted(p for p in pos if 0 <= p < S)


@pytest.mark.parametrize("name", ["gemma2_local_w4096_cap50", "gemma2_local_w4096_cap0",
                                  "packed_varlen_cap30", "sink_gqa64_cap0", "sink_gqa64_cap30",
                                  "long_noncausal_16k_cap50", "long_causal_32k_cap50",
                                  "decode_sq128_sk32k_cap30_sink", "hd512_cap30",
                                  "gemma2_local_w4096_cap50_bias"])
def test_fullsize_sampled(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    gpu = run_gpu(w, inp, kv_splits=w.kv_splits)
    tol = TOL[w.dtype]
    g = w.Hkv - 1
    G = w.Hq // w.Hkv
    heads = list(range(g * G, (g + 1) * G))
    batches = list(range(w.B)) if w.sink else [w.B - 1]
    p = problem_from_inputs(w, inp, heads=[g], batches=batches)
    O, LSE = oracle.forward(p)
    seg_row = None if inp["seg"] is None else inp["seg"][batches[-1]].numpy()
    rows = sample_positions(w.Sq, seg_row)
    cols = sample_positions(w.Sk, seg_row) if w.Sq == w.Sk else sample_positions(w.Sk)
    ref = oracle.backward(p, to64(inp["dO"])[batches][:, :, heads], O, LSE, rows=rows, cols=cols)
    Og = to64(gpu["O"])[batches][:, :, heads]
    errs = {"O": frob_rel(Og, O)}
    Lg = to64(gpu["LSE"])[batches][:, heads]
    errs["LSE"] = frob_rel(Lg, LSE)
    errs["dq"] = frob_rel(to64(gpu["dq"])[batches][:, rows][:, :, heads], ref["dq"][:, rows])
    errs["dk"] = frob_rel(to64(gpu["dk"])[batches][:, cols][:, :, [g]], ref["dk"][:, cols])
    errs["dv"] = frob_rel(to64(gpu["dv"])[batches][:, cols][:, :, [g]], ref["dv"][:, cols])
    if w.sink:
        errs["dsink"] = frob_rel(gpu["dsink"].double().cpu().numpy()[heads], ref["dsink"])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (name, errs)


def test_fullsize_thd_prefix_sampled():
    """The packed chunked-prefill workload through cu_seqlens / cu_seqlens_k as bench.py runs
    it, checked on its second sequence (every row of O / LSE, sampled dQ rows and dK / dV
    columns, one kv group) against the oracle on that sequence alone."""
    w = WORKLOADS["thd_prefix_cap30"]
    inp = make_inputs(w)
    cq, ck = inp["cu_q"], inp["cu_k"]
    gpu = run_gpu(w, inp, cu_seqlens=cq.cuda(), cu_seqlens_k=ck.cuda())
    q0, q1, k0, k1 = int(cq[1]), int(cq[2]), int(ck[1]), int(ck[2])
    g = w.Hkv - 1
    G = w.Hq // w.Hkv
    heads = list(range(g * G, (g + 1) * G))
    p = oracle.Problem(to64(inp["q"])[:, q0:q1][:, :, heads], to64(inp["k"])[:, k0:k1][:, :, [g]],
                       to64(inp["v"])[:, k0:k1][:, :, [g]], scale=w.scale, causal=w.causal,
                       window=w.window, softcap=w.softcap)
    O, LSE = oracle.forward(p)
    rows, cols = sample_positions(q1 - q0), sample_positions(k1 - k0)
    ref = oracle.backward(p, to64(inp["dO"])[:, q0:q1][:, :, heads], O, LSE, rows=rows, cols=cols)
    sl = lambda x: x[:, q0:q1][:, :, heads]  # noqa: E731
    errs = {"O": frob_rel(sl(to64(gpu["O"])), O),
            "LSE": frob_rel(to64(gpu["LSE"])[:, heads][:, :, q0:q1], LSE),
            "dq": frob_rel(sl(to64(gpu["dq"]))[:, rows], ref["dq"][:, rows]),
            "dk": frob_rel(to64(gpu["dk"])[:, k0:k1][:, cols][:, :, [g]], ref["dk"][:, cols]),
            "dv": frob_rel(to64(gpu["dv"])[:, k0:k1][:, cols][:, :, [g]], ref["dv"][:, cols])}
    bad = {k: v for k, v in errs.items() if not v <= TOL[w.dtype]}
    assert not bad, errs
    # keys past the last sequence belong to no query: zero gradients
    assert int(ck[-1]) < w.Sk and gpu["dk"][:, int(ck[-1]):].abs().max().item() == 0.0
