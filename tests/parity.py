"""Helpers for the GPU parity tests: run the CUDA path through the binding and the fp64
oracle on the same seeded inputs, and compare them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import Workload, make_inputs

# Max Frobenius-relative error, per input dtype.
TOL = {"f32": 1e-5, "bf16": 1e-2}


def frob_rel(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def to64(t):
    return None if t is None else t.detach().to("cpu", torch.float32).double().numpy()


def problem_from_inputs(w: Workload, inp: dict, heads=None, batches=None) -> oracle.Problem:
    """Oracle problem on the exact (upcast) inputs; optionally restricted to whole kv groups
    ``heads`` (kv head indices) and batches."""
    q, k, v = to64(inp["q"]), to64(inp["k"]), to64(inp["v"])
    bias = inp["bias"]  # sliced before it is upcast: at full size it is a few GB in bf16
    sink = None if inp["sink"] is None else inp["sink"].double().numpy()
    seg = None if inp["seg"] is None else inp["seg"].numpy()
    if batches is not None:
        q, k, v = q[batches], k[batches], v[batches]
        seg = None if seg is None else seg[batches]
        if bias is not None and bias.shape[0] > 1:
            bias = bias[batches]
    if heads is not None:
        G = w.Hq // w.Hkv
        qh = np.concatenate([np.arange(g * G, (g + 1) * G) for g in heads])
        q, k, v = q[:, :, qh], k[:, :, heads], v[:, :, heads]
        sink = None if sink is None else sink[qh]
        if bias is not None and bias.shape[1] > 1:
            bias = bias[:, torch.as_tensor(qh)]
    return oracle.Problem(q, k, v, scale=w.scale, causal=w.causal, window=w.window,
                          softcap=w.softcap, bias=to64(bias), sink=sink, seg_q=seg, seg_k=seg)


def run_gpu(w: Workload, inp: dict, dev="cuda", **extra):
    import attention_flash_attn_gb300 as fa
    t = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    kw = dict(causal=w.causal, window=w.window, softcap=w.softcap, sink=t["sink"],
              scale=w.scale, bias=t["bias"], seg_q=t["seg"], seg_k=t["seg"])
    kw.update(extra)
    O, LSE = fa.attn_fwd(t["q"], t["k"], t["v"], **kw)
    dQ, dK, dV, dbias, dsink = fa.attn_bwd(t["q"], t["k"], t["v"], O, LSE, t["dO"], **kw)
    torch.cuda.synchronize()
    assert fa.attn_check_device_status() == 0
    return {"O": O, "LSE": LSE, "dq": dQ, "dk": dK, "dv": dV, "dbias": dbias, "dsink": dsink}


def varlen_oracle(w: Workload, inp: dict, cu_q, cu_k):
    """thd varlen: every sequence is an attention problem of its own (B = 1, its own query and
    key lengths, bottom-right causal / window alignment) -- the oracle run per sequence, its
    outputs placed back at the sequence's tokens.  Tokens past the last boundary form one more
    sequence; a sequence without keys keeps O = 0 and LSE = its sink (or -inf)."""
    q, k, v, dO = to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), to64(inp["dO"])
    sink = None if inp["sink"] is None else inp["sink"].double().numpy()
    bq, bk = list(cu_q) + [w.Sq], list(cu_k) + [w.Sk]
    O, dq = np.zeros_like(q), np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    LSE = np.full((1, w.Hq, w.Sq), -np.inf)
    dsink = None if sink is None else np.zeros(w.Hq)
    for s in range(len(bq) - 1):
        q0, q1, k0, k1 = bq[s], bq[s + 1], bk[s], bk[s + 1]
        if q1 == q0:
            continue
        if k1 == k0:
            if sink is not None:
                LSE[0, :, q0:q1] = sink[:, None]
            continue
        p = oracle.Problem(q[:, q0:q1], k[:, k0:k1], v[:, k0:k1], scale=w.scale, causal=w.causal,
                           window=w.window, softcap=w.softcap, sink=sink)
        Os, Ls = oracle.forward(p)
        g = oracle.backward(p, dO[:, q0:q1], Os, Ls)
        O[:, q0:q1], LSE[:, :, q0:q1] = Os, Ls
        dq[:, q0:q1], dk[:, k0:k1], dv[:, k0:k1] = g["dq"], g["dk"], g["dv"]
        if sink is not None:
            dsink += g["dsink"]
    return {"O": O, "LSE": LSE, "dq": dq, "dk": dk, "dv": dv, "dbias": None, "dsink": dsink}


def full_oracle(w: Workload, inp: dict):
    p = problem_from_inputs(w, inp)
    O, LSE = oracle.forward(p)
    g = oracle.backward(p, to64(inp["dO"]), O, LSE)
    g["O"], g["LSE"] = O, LSE
    return g


def compare_full(w: Workload, gpu: dict, ref: dict) -> dict:
    """Frobenius-relative errors of every output against the oracle."""
    errs = {}
    for key in ("O", "dq", "dk", "dv", "dbias", "dsink"):
        if ref.get(key) is None:
            assert gpu.get(key) is None, key
            continue
        errs[key] = frob_rel(to64(gpu[key]), ref[key])
    lse_g = to64(gpu["LSE"])
    fin = np.isfinite(ref["LSE"])
    assert np.array_equal(np.isfinite(lse_g), fin), "LSE -inf pattern differs"
    errs["LSE"] = frob_rel(lse_g[fin], ref["LSE"][fin]) if fin.any() else 0.0
    return errs


def check_against_oracle_small(w: Workload, **extra):
    """Run a small workload through the binding and assert every output is within the
    dtype's tolerance of the fp64 oracle; returns the errors."""
    inp = make_inputs(w)
    errs = compare_full(w, run_gpu(w, inp, **extra), full_oracle(w, inp))
    bad = {k: v for k, v in errs.items() if not v <= TOL[w.dtype]}
    assert not bad, (w.name, errs)
    return errs
