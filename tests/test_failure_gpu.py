"""The kernels' failure path on the GPU, without any fault: a bounded wait that gives up by
design (attn_selftest_wait_expiry waits on an mbarrier that nothing completes), the status
words it leaves, the early return of later kernels while the status bit is set, and a normal
call afterwards on the same context.  A malformed cu_seqlens (every value inside [0, Sq],
only the order broken, so every access stays inside its array) is reported the same way.
Every failure here is made on purpose and ends with a status the host reads; nothing traps,
faults or hangs (TransformerEngine PR #3391, "What changed": fail closed)."""
import ctypes
import time

import pytest
import torch

from parity import check_against_oracle_small
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

ATTN_ERR_DEVICE = 5


def _words(ws):
    return [int(x) & 0xFFFFFFFF for x in ws.view(torch.int32).cpu().tolist()]


def test_bounded_wait_gives_up_records_and_the_context_stays_usable():
    import attention_flash_attn_gb300 as fa
    L = fa.lib()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert L.attn_selftest_wait_expiry(ws.data_ptr(), ws.numel(), 20_000_000, st) == 0
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    w = _words(ws)
    assert w[0] & 1  # kStatusWaitTimeout
    assert w[1] == 1  # the first timeout was recorded ...
    assert w[2] == w[48] and w[3] == 0  # ... on barrier A, parity 0
    assert w[4] == 0 and w[5] == 0 and w[6] == 0  # CTA 0, thread 0
    assert w[10] == w[49] and w[11] == 0x100  # warp 1 of that CTA gave up on barrier B
    assert elapsed < 1.5, elapsed  # the others left on the status bit, not on their own 2 s limit
    assert L.attn_check_device_status(ws.data_ptr(), st) == ATTN_ERR_DEVICE
    assert _words(ws)[0] == 0  # read and cleared
    assert L.attn_check_device_status(ws.data_ptr(), st) == 0
    # the same context still computes correctly
    check_against_oracle_small(Workload("after_selftest", "bf16", B=1, Sq=200, Sk=200, Hq=2, Hkv=1, D=64,
                                        causal=True, softcap=30.0, sink=True))


def test_kernels_return_at_once_while_the_status_bit_is_set():
    """With the timeout bit already in its workspace (set from the host), attn_fwd's kernels
    leave O untouched; once attn_check_device_status has read and cleared it, the same call
    computes O."""
    import attention_flash_attn_gb300 as fa
    from attention_flash_attn_gb300 import build_args
    L = fa.lib()
    w = Workload("sticky", "bf16", B=1, Sq=256, Sk=256, Hq=2, Hkv=1, D=128, causal=True, softcap=30.0)
    inp = make_inputs(w)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    a, keep = build_args(t["q"], t["k"], t["v"], causal=True, softcap=30.0, scale=w.scale)
    need = L.attn_fwd_workspace_size(ctypes.byref(a))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[0] = 1
    O = torch.full((1, 256, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    LSE = torch.full((1, 2, 256), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.attn_fwd(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), ws.data_ptr(), need, st) == 0
    torch.cuda.synchronize()
    assert torch.isnan(O).all() and torch.isnan(LSE).all()
    assert L.attn_check_device_status(ws.data_ptr(), st) == ATTN_ERR_DEVICE
    assert L.attn_fwd(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), ws.data_ptr(), need, st) == 0
    assert L.attn_check_device_status(ws.data_ptr(), st) == 0
    ref, _ = fa.attn_fwd(t["q"], t["k"], t["v"], causal=True, softcap=30.0, scale=w.scale)
    assert torch.equal(O, ref)
    del keep


def test_malformed_cu_seqlens_reported_through_the_status_word():
    """cu_seqlens whose values all lie in [0, Sq] but out of order: the call is accepted (the
    host cannot read device memory before launching) and the metadata kernel records the error;
    the next well-formed call reports nothing."""
    import attention_flash_attn_gb300 as fa
    w = Workload("bad_cu", "bf16", B=1, Sq=515, Sk=515, Hq=2, Hkv=1, D=64, causal=True, softcap=20.0)
    inp = make_inputs(w)
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    bad = torch.tensor([0, 300, 100, 515], dtype=torch.int32, device="cuda")
    good = torch.tensor([0, 100, 300, 515], dtype=torch.int32, device="cuda")
    fa.attn_fwd(t["q"], t["k"], t["v"], causal=True, softcap=20.0, cu_seqlens=bad)
    assert fa.attn_check_device_status() == ATTN_ERR_DEVICE
    fa.attn_fwd(t["q"], t["k"], t["v"], causal=True, softcap=20.0, cu_seqlens=good)
    assert fa.attn_check_device_status() == 0
