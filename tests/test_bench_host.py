"""Host logic of bench.py: the visible-pair count that the flop figures rest on equals the
oracle's brute-force count of the mask definition."""
import numpy as np
import pytest

import oracle
from bench import flops, host_cpu, memory_phase_bytes, visible_pairs
from workloads import WORKLOADS, Workload, make_inputs


@pytest.mark.parametrize("w", [
    Workload("a", "bf16", B=2, Sq=97, Sk=97, Hq=3, Hkv=1, D=8, causal=True),
    Workload("b", "bf16", B=1, Sq=97, Sk=97, Hq=2, Hkv=2, D=8, causal=True, window=20),
    Workload("c", "bf16", B=1, Sq=60, Sk=90, Hq=1, Hkv=1, D=8, causal=True),
    Workload("d", "bf16", B=1, Sq=80, Sk=80, Hq=1, Hkv=1, D=8, causal=False, window=9),
    Workload("e", "bf16", B=3, Sq=150, Sk=150, Hq=2, Hkv=1, D=8, causal=True, segments=True,
             run_lo=5, run_hi=40),
], ids=lambda w: w.name)
def test_visible_pairs_matches_oracle_brute_force(w):
    seg = make_inputs(w)["seg"]
    z = np.zeros
    p = oracle.Problem(z((w.B, w.Sq, w.Hq, 1)), z((w.B, w.Sk, w.Hkv, 1)), z((w.B, w.Sk, w.Hkv, 1)),
                       scale=1.0, causal=w.causal, window=w.window,
                       seg_q=None if seg is None else seg.numpy())
    assert visible_pairs(w, None if seg is None else seg.numpy()) == oracle.count_visible(p)


def test_thd_visible_pairs_match_per_sequence_oracle_counts():
    """thd varlen: the count over (cu_q, cu_k) bounds equals the oracle's brute-force count run
    on each sequence as its own problem (bottom-right causal / window inside it), including the
    trailing sequence past the last bounds."""
    w = WORKLOADS["thd_prefix_cap30"].replace(Sq=300, Sk=700, Hq=2, Hkv=1, run_lo=20, run_hi=90,
                                              prefix_hi=200, window=37)
    inp = make_inputs(w)
    cq = [int(x) for x in inp["cu_q"]] + [w.Sq]
    ck = [int(x) for x in inp["cu_k"]] + [w.Sk]
    z = np.zeros
    ref = 0
    for s in range(len(cq) - 1):
        lq, lk = cq[s + 1] - cq[s], ck[s + 1] - ck[s]
        if lq and lk:
            p = oracle.Problem(z((1, lq, w.Hq, 1)), z((1, lk, w.Hkv, 1)), z((1, lk, w.Hkv, 1)), scale=1.0,
                               causal=w.causal, window=w.window)
            ref += oracle.count_visible(p)
    assert visible_pairs(w, None, (inp["cu_q"], inp["cu_k"])) == ref > 0


def test_headline_flop_counts():
    w = WORKLOADS["gemma2_local_w4096_cap50"]
    # causal with a 4096 window over 8192 tokens: 4096*4097/2 + 4096*4096 pairs per (b, h)
    per = 4096 * 4097 // 2 + 4096 * 4096
    assert visible_pairs(w, None) == per * w.B * w.Hq
    assert flops(w, None, "fwdbwd") == per * w.B * w.Hq * 14 * 256
    w5 = WORKLOADS["long_causal_32k_cap50"]
    assert visible_pairs(w5, None) == 32768 * 32769 // 2 * 32


def test_memory_phase_bytes():
    """K3 / K5 bytes of the headline workload, written out term by term: O and dO read (bf16),
    LSE read, D and LSE*log2(e) written (fp32, rows padded to 128), the fp32 dQ accumulator
    zeroed (K3); the accumulator read and dQ written (K5).  Head dim 128 adds -D's 16-byte
    bf16 parts per row; the FFMA path (fp32) has no accumulator; a bias adds its fp32
    accumulator read and its own dtype written."""
    w = WORKLOADS["gemma2_local_w4096_cap50"]
    elems, rows = 2 * 8192 * 16 * 256, 2 * 16 * 8192
    b = memory_phase_bytes(w, "tc", 0, 0)
    assert b["K3"] == 2 * elems * 2 + rows * 4 + rows * 4 + rows * 4 + elems * 4
    assert b["K5"] == elems * 4 + elems * 2
    assert b["K1"] == 0
    w3 = WORKLOADS["packed_varlen_cap30"]
    e3, r3 = 4 * 8192 * 8 * 128, 4 * 8 * 8192
    b3 = memory_phase_bytes(w3, "tc", 4096, 0)
    assert b3["K3"] == 2 * e3 * 2 + 3 * r3 * 4 + 16 * r3 + 4 * e3
    assert b3["K1"] == 4 * 4 * (8192 + 8192) + 4096
    f = Workload("f", "f32", B=1, Sq=100, Sk=100, Hq=2, Hkv=2, D=64, causal=True)
    w5 = WORKLOADS["hd512_cap30"]  # the wide form: no fp32 dQ accumulator, dQ written by its GEMM
    e5, r5 = 2048 * 8 * 512, 8 * 2048
    b5 = memory_phase_bytes(w5, "tc", 0, 0)
    assert b5["K3"] == 2 * e5 * 2 + 3 * r5 * 4 and b5["K5"] == 0
    bf = memory_phase_bytes(f, "simt", 0, 7)
    assert bf["K3"] == 2 * 100 * 2 * 64 * 4 + 200 * 4 + 256 * 4  # D's rows padded to 128 per head
    assert bf["K5"] == 7 * 8


def test_clock_samples_are_taken_inside_the_timed_region(tmp_path):
    """Only nvidia-smi samples whose timestamps fall in the timed region's wall-clock window
    count (the idle ones before and after are dropped); throttle reasons come from those."""
    import datetime
    import time

    import bench

    c = bench.ClockSampler(0)
    now = time.time()
    ts = lambda t: datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]  # noqa: E731
    idle = "0x0, Not Active, Not Active, Not Active, Not Active"
    rows = [f"{ts(now - 1.0)}, 0, 1200, 2070, 300.0, {idle}",
            f"{ts(now + 0.01)}, 0, 2070, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Active",
            f"{ts(now + 0.03)}, 0, 2040, 2070, 1350.0, 0x0, Not Active, Not Active, Not Active, Active",
            f"{ts(now + 2.0)}, 0, 1000, 2070, 200.0, {idle}"]
    c.out.write("\n".join(rows) + "\n")
    c.out.flush()

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    c.proc = Done()
    c.mark(now, now + 0.05)
    clk = c.stop()
    assert clk == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}


def test_host_cpu_names_the_processor():
    """The oracle's timings name the host processor: the machine type, then a model name or
    the ARM implementer / part codes."""
    import platform
    name = host_cpu()
    assert name.startswith(platform.machine())
    assert len(name) > len(platform.machine())



@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_bench_call_arguments_pass_the_binding_checks(name):
    """Every bench workload's arguments (shapes of q / k / v, ids, boundaries, sink, bias, a
    metadata buffer of the size the library asks for) pass the binding's checks; the workload
    is cut to at most 1024 query rows (the checks depend on shapes, not sizes)."""
    import ctypes
    import attention_flash_attn_gb300 as fa
    from bench import call_kwargs
    w = WORKLOADS[name]
    sq = min(w.Sq, 1024)
    w = w.replace(Sq=sq, Sk=w.Sk * sq // w.Sq, run_lo=min(w.run_lo, 32), run_hi=min(w.run_hi, 256),
                  prefix_hi=min(w.prefix_hi, 256))
    t = make_inputs(w)
    kw = call_kwargs(w, t)
    a, keep = fa.build_args(t["q"], t["k"], t["v"], **kw)
    need = fa.lib().attn_meta_size(ctypes.byref(a))
    assert (need > 0) == (w.segments or w.thd_prefix)
    if need:  # a buffer of that size at a 256-byte boundary, as a device allocation would be
        import torch
        raw = torch.zeros(need + 256, dtype=torch.uint8)
        off = -raw.data_ptr() % 256
        a, keep = fa.build_args(t["q"], t["k"], t["v"], meta=raw[off:off + need], **kw)
    assert fa.lib().attn_fwd_workspace_size(ctypes.byref(a)) > 0
    assert fa.lib().attn_bwd_workspace_size(ctypes.byref(a)) > 0
