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
