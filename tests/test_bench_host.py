"""Host logic of bench.py: the visible-pair count that the flop figures rest on equals the
oracle's brute-force count of the mask definition."""
import numpy as np
import pytest

import oracle
from bench import flops, visible_pairs
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


def test_headline_flop_counts():
    w = WORKLOADS["gemma2_local_w4096_cap50"]
    # causal with a 4096 window over 8192 tokens: 4096*4097/2 + 4096*4096 pairs per (b, h)
    per = 4096 * 4097 // 2 + 4096 * 4096
    assert visible_pairs(w, None) == per * w.B * w.Hq
    assert flops(w, None, "fwdbwd") == per * w.B * w.Hq * 14 * 256
    w5 = WORKLOADS["long_causal_32k_cap50"]
    assert visible_pairs(w5, None) == 32768 * 32769 // 2 * 32
