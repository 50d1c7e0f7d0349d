"""attn_fwd_noalloc: the forward for callers that cannot allocate device memory (plugins
hosted by a runtime that owns every device allocation, fixed-budget deployments).  Its
scratch is an array compiled into the library, so these tests check that it gives the same
results as attn_fwd with a caller-provided workspace, on two calls in a row (the second call
sees the first call's leftovers in the shared array), and that an over-size request is turned
away before anything runs.

This file is collected last on purpose: if it fails, every other test has already run.
"""
import ctypes

import pytest
import torch

from parity import TOL, frob_rel, to64
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc_fwd(fa, t, w, **kw):
    a, keep = fa.build_args(t["q"], t["k"], t["v"], causal=w.causal, window=w.window, softcap=w.softcap,
                            sink=t["sink"], scale=w.scale, **kw)
    B, Sq, Hq, D = t["q"].shape
    O = torch.full((B, Sq, Hq, D), float("nan"), dtype=t["q"].dtype, device="cuda")
    LSE = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    status = fa.lib().attn_fwd_noalloc(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), st)
    torch.cuda.synchronize()
    del keep
    return status, O, LSE


def test_noalloc_forward_matches_workspace_forward_twice():
    import attention_flash_attn_gb300 as fa
    cases = [
        # packed segments (scratch holds the segment metadata), GQA, sink, cap
        (Workload("noalloc_packed", "bf16", B=2, Sq=700, Sk=700, Hq=4, Hkv=2, D=128, causal=True,
                  softcap=30.0, q_std=3.0, sink=True, segments=True, run_lo=40, run_hi=300), {}),
        # different shapes and masks on the second call: cu_seqlens, head dim 64, window
        (Workload("noalloc_cu", "bf16", B=1, Sq=515, Sk=515, Hq=2, Hkv=1, D=64, causal=True,
                  window=200, softcap=20.0), {"cu": [0, 100, 333, 515]}),
    ]
    for w, extra in cases:
        inp = make_inputs(w)
        t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
        kw = {}
        if "cu" in extra:
            kw["cu_seqlens"] = torch.tensor(extra["cu"], dtype=torch.int32, device="cuda")
        else:
            kw["seg_q"] = t["seg"]
        ref_O, ref_LSE = fa.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, window=w.window,
                                     softcap=w.softcap, sink=t["sink"], scale=w.scale, **kw)
        status, O, LSE = _noalloc_fwd(fa, t, w, **kw)
        assert status == 0, fa.lib().attn_status_string(status)
        assert frob_rel(to64(O), to64(ref_O)) <= TOL[w.dtype], w.name
        fin = torch.isfinite(ref_LSE)
        assert torch.equal(torch.isfinite(LSE), fin)
        assert frob_rel(to64(LSE[fin]), to64(ref_LSE[fin])) <= TOL[w.dtype], w.name


def test_noalloc_rejects_requests_beyond_its_array():
    import attention_flash_attn_gb300 as fa
    from attention_flash_attn_gb300 import _capi
    a = _capi.AttnArgs()
    S = 1 << 20  # cu_seqlens ids alone need 4 MiB of scratch
    a.dtype, a.B, a.Sq, a.Sk, a.Hq, a.Hkv, a.D = 1, 1, S, S, 1, 1, 64
    a.q = a.k = a.v = 0x10000
    a.q_stride_b = a.k_stride_b = a.v_stride_b = S * 64
    a.q_stride_s = a.k_stride_s = a.v_stride_s = 64
    a.q_stride_h = a.k_stride_h = a.v_stride_h = 64
    a.cu_seqlens, a.nseq = 0x20000, 1
    a.scale = 0.125
    L = fa.lib()
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) > (4 << 20)
    n = L.attn_launch_counter()
    assert L.attn_fwd_noalloc(ctypes.byref(a), 0x30000, 0x40000, None) == _capi.ATTN_ERR_WORKSPACE
    assert L.attn_launch_counter() == n


def test_noalloc_device_errors_can_be_read_back():
    """attn_noalloc_check_device_status reads the status word of the built-in array: a
    cu_seqlens whose values all lie in [0, Sq] but out of order (every access stays inside
    its array) is reported as a device-side error of that call; the next well-formed call
    reports nothing and matches attn_fwd."""
    import attention_flash_attn_gb300 as fa
    from attention_flash_attn_gb300 import _capi
    L = fa.lib()
    w = Workload("noalloc_bad_cu", "bf16", B=1, Sq=515, Sk=515, Hq=2, Hkv=1, D=64, causal=True, softcap=20.0)
    inp = make_inputs(w)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    st = torch.cuda.current_stream().cuda_stream
    bad = torch.tensor([0, 300, 100, 515], dtype=torch.int32, device="cuda")
    good = torch.tensor([0, 100, 300, 515], dtype=torch.int32, device="cuda")
    status, _, _ = _noalloc_fwd(fa, t, w, cu_seqlens=bad)
    assert status == 0
    assert L.attn_noalloc_check_device_status(st) == _capi.ATTN_ERR_DEVICE
    assert L.attn_noalloc_check_device_status(st) == 0
    status, O, LSE = _noalloc_fwd(fa, t, w, cu_seqlens=good)
    assert status == 0
    assert L.attn_noalloc_check_device_status(st) == 0
    ref_O, ref_LSE = fa.attn_fwd(t["q"], t["k"], t["v"], causal=True, softcap=20.0, scale=w.scale,
                                 cu_seqlens=good)
    assert frob_rel(to64(O), to64(ref_O)) <= TOL[w.dtype]


# Child program: the forward in contexts of the caller's own (driver API), the way a plugin
# hosted by another runtime calls it.  It makes a context, runs attn_fwd_noalloc there on packed
# segments (the array then holds the segment metadata), destroys the context, makes a second
# one and runs the same call: the array lives at a new address in the new context, and both
# calls must give the same O and LSE, which must also match a float64 softmax of the same
# bf16-rounded inputs.  Torch's CUDA state is never touched in the child.
_CONTEXT_CHILD = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from attention_flash_attn_gb300 import _capi

cu = ctypes.CDLL("libcuda.so.1")
def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what}: CUresult {r}")
ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")

B, S, H, D = 1, 300, 2, 64
rng = np.random.default_rng(7)
def bf16(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r, (r.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
q16, q = bf16(rng.normal(0, 2, (B, S, H, D)))
k16, k = bf16(rng.normal(0, 2, (B, S, H, D)))
v16, v = bf16(rng.normal(0, 1, (B, S, H, D)))
seg = np.repeat(np.arange(4, dtype=np.int32), [70, 101, 29, 100]).reshape(B, S)
scale, cap = 0.125, 20.0

def run():
    ctx = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate")
    bufs = []
    def up(a):
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(a.nbytes)), "cuMemAlloc")
        ck(cu.cuMemcpyHtoD_v2(p, a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)), "HtoD")
        bufs.append(p)
        return p.value
    O = np.zeros((B, S, H, D), np.uint16)
    L = np.zeros((B, H, S), np.float32)
    a = _capi.AttnArgs()
    a.dtype, a.B, a.Sq, a.Sk, a.Hq, a.Hkv, a.D = _capi.ATTN_DTYPE_BF16, B, S, S, H, H, D
    st = (S * H * D, H * D, D)
    a.q, a.k, a.v = up(q16), up(k16), up(v16)
    a.q_stride_b, a.q_stride_s, a.q_stride_h = st
    a.k_stride_b, a.k_stride_s, a.k_stride_h = st
    a.v_stride_b, a.v_stride_s, a.v_stride_h = st
    a.seg_q = a.seg_k = up(seg)
    a.causal, a.softcap, a.scale = 1, cap, scale
    dO, dL = up(O), up(L)
    lib = _capi.lib()
    s = lib.attn_fwd_noalloc(ctypes.byref(a), dO, dL, None)
    if s != 0:
        raise SystemExit(f"attn_fwd_noalloc: {s}")
    ck(cu.cuCtxSynchronize(), "sync")
    s = lib.attn_noalloc_check_device_status(None)
    if s != 0:
        raise SystemExit(f"status: {s}")
    ck(cu.cuMemcpyDtoH_v2(O.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(dO), ctypes.c_size_t(O.nbytes)), "DtoH")
    ck(cu.cuMemcpyDtoH_v2(L.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(dL), ctypes.c_size_t(L.nbytes)), "DtoH")
    for p in bufs:
        ck(cu.cuMemFree_v2(p), "cuMemFree")
    ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
    return (O.astype(np.uint32) << 16).view(np.float32), L

O1, L1 = run()
O2, L2 = run()
assert np.array_equal(O1, O2) and np.array_equal(L1, L2), "the two contexts disagree"
# float64 softmax of the same inputs: scale, cap, causal mask within equal segment ids
i, j = np.arange(S)[:, None], np.arange(S)[None, :]
vis = (j <= i) & (seg[0][:, None] == seg[0][None, :])
err = 0.0
for h in range(H):
    u = scale * q[0, :, h] @ k[0, :, h].T
    t = np.where(vis, cap * np.tanh(u / cap), -np.inf)
    m = t.max(1, keepdims=True)
    p = np.exp(t - m)
    o = (p @ v[0, :, h]) / p.sum(1, keepdims=True)
    err = max(err, np.linalg.norm(O1[0, :, h] - o) / np.linalg.norm(o))
    lse = (m[:, 0] + np.log(p.sum(1))).astype(np.float64)
    err = max(err, np.abs(L1[0, h] - lse).max() / np.abs(lse).max())
assert err < 1e-2, err
print("ok", err)
'''


def test_noalloc_in_contexts_of_the_caller_s_own():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CONTEXT_CHILD, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.stdout[-2000:], r.stderr[-4000:])
