"""Seeded synthetic workloads for the softcap / sink attention path.

This module holds shapes and random draws only -- none of the method's
arithmetic.  Both the CUDA path (through ``bench.py`` and the GPU tests) and the
fp64 oracle read their inputs from here, so the two always see the same numbers.

Draw order (one ``torch.Generator`` on the CPU, seeded once per workload):
q, k, v, dO, bias, sink, segment runs; each draw is fp32 N(0,1) scaled by the
workload's standard deviation and then cast to the workload dtype.

The workloads are the ones the softcap / sink pages motivate (a Gemma2-style local
layer with a cap of 50, packed variable-length rows with a cap of 30, a learnable
sink with offsets drawn as randn x 5, a long-context causal stress case) plus one
tiny fp32 case with an additive bias that the oracle finishes in seconds.  No
public dataset or benchmark suite is involved: the inputs are synthetic by design.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str               # "f32" or "bf16"
    B: int
    Sq: int
    Sk: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    window: int = 0          # 0: no sliding window
    softcap: float = 0.0     # 0: no cap
    q_std: float = 1.0       # std of q and k
    v_std: float = 1.0       # std of v and dO
    bias: bool = False       # post-scale additive bias ~ N(0,1) [1|B, 1|Hq, Sq, Sk] (bias_dims)
    bias_dims: str = "h"     # dimensions the bias has of its own: "h" [1,Hq], "b" [B,1], "bh", ""
    sink: bool = False       # per-query-head sink offsets ~ randn * 5
    segments: bool = False   # packed rows: run lengths ~ U[run_lo, run_hi], last truncated
    run_lo: int = 64
    run_hi: int = 4096
    seed: int = 0
    kv_splits: int = 0       # split-KV forward: key shares per query tile (0: off)
    # thd varlen with cached prefixes (B = 1): query runs ~ U[run_lo, run_hi] over Sq (last
    # truncated); sequence s holds a cached prefix ~ U[0, prefix_hi] of keys before its own
    # query tokens' keys (keys = prefix + queries, bottom-right causal), until Sk is used up;
    # left-over keys form a trailing sequence without queries.
    thd_prefix: bool = False
    prefix_hi: int = 2048

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return {"f32": torch.float32, "bf16": torch.bfloat16}[self.dtype]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The full-size workloads (the first is the tiny fp32 correctness case).
WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_f32_softcap_bias", "f32", B=1, Sq=256, Sk=256, Hq=2, Hkv=2, D=64,
                 causal=True, softcap=30.0, q_std=4.0, bias=True),
        Workload("gemma2_local_w4096_cap50", "bf16", B=2, Sq=8192, Sk=8192, Hq=16, Hkv=8, D=256,
                 causal=True, window=4096, softcap=50.0, q_std=3.0),
        Workload("gemma2_local_w4096_cap0", "bf16", B=2, Sq=8192, Sk=8192, Hq=16, Hkv=8, D=256,
                 causal=True, window=4096, softcap=0.0, q_std=3.0),
        # The same layer with a post-scale additive bias per query head ([1, Hq, S, S] bf16):
        # the bias path of the tensor-core kernels (this build's own workload).
        Workload("gemma2_local_w4096_cap50_bias", "bf16", B=2, Sq=8192, Sk=8192, Hq=16, Hkv=8, D=256,
                 causal=True, window=4096, softcap=50.0, q_std=3.0, bias=True),
        Workload("packed_varlen_cap30", "bf16", B=4, Sq=8192, Sk=8192, Hq=8, Hkv=8, D=128,
                 causal=True, softcap=30.0, q_std=3.0, segments=True),
        Workload("sink_gqa64_cap0", "bf16", B=2, Sq=4096, Sk=4096, Hq=64, Hkv=8, D=64,
                 causal=True, softcap=0.0, sink=True),
        Workload("sink_gqa64_cap30", "bf16", B=2, Sq=4096, Sk=4096, Hq=64, Hkv=8, D=64,
                 causal=True, softcap=30.0, sink=True),
        Workload("long_causal_32k_cap50", "bf16", B=1, Sq=32768, Sk=32768, Hq=32, Hkv=16, D=256,
                 causal=True, softcap=50.0, q_std=3.0),
        Workload("long_noncausal_16k_cap50", "bf16", B=1, Sq=16384, Sk=16384, Hq=32, Hkv=16, D=256,
                 causal=False, softcap=50.0, q_std=3.0),
        # Decode-like rows for the split-KV forward: one 128-row query tile per head against
        # 32k keys (bottom-right causal), too few query tiles to fill the GPU unsplit.
        Workload("decode_sq128_sk32k_cap30_sink", "bf16", B=1, Sq=128, Sk=32768, Hq=32, Hkv=8, D=128,
                 causal=True, softcap=30.0, q_std=3.0, sink=True, kv_splits=4),
        # Head dim above 256 (the FFMA kernels; the pages' chunked head-dim accumulation).
        Workload("hd512_cap30", "bf16", B=1, Sq=2048, Sk=2048, Hq=8, Hkv=4, D=512, causal=True,
                 softcap=30.0, q_std=2.0),
        # Chunked prefill against a KV cache, packed thd: per sequence a query chunk and its
        # keys (cached prefix + the chunk), Sq != Sk per sequence, bottom-right causal.
        Workload("thd_prefix_cap30", "bf16", B=1, Sq=8192, Sk=20480, Hq=8, Hkv=8, D=128,
                 causal=True, softcap=30.0, q_std=3.0, thd_prefix=True, run_lo=64, run_hi=2048),
    ]
}


def segment_runs(gen: torch.Generator, B: int, S: int, lo: int, hi: int, tile: int = 128):
    """Segment ids [B,S] int32 from run lengths ~ U[lo,hi] per row, last run truncated.

    Ids are increasing within a row (0, 1, 2, ...).  The whole draw is repeated until at
    least one run boundary inside some row is not a multiple of ``tile``.
    """
    while True:
        rows, unaligned = [], False
        for _ in range(B):
            lens, total = [], 0
            while total < S:
                L = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
                L = min(L, S - total)
                lens.append(L)
                total += L
                if total < S and total % tile != 0:
                    unaligned = True
            rows.append(torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32),
                                                torch.tensor(lens)))
        if unaligned:
            return torch.stack(rows).to(torch.int32)


def thd_prefix_bounds(gen: torch.Generator, Sq: int, Sk: int, lo: int, hi: int, prefix_hi: int):
    """Query and key boundaries (cu_q, cu_k, int32 [nseq + 1]) of a packed chunked-prefill
    batch: query runs ~ U[lo, hi] (last truncated to Sq), each sequence's keys a prefix
    ~ U[0, prefix_hi] plus its queries; sequences stop where the keys would pass Sk."""
    cu_q, cu_k = [0], [0]
    while cu_q[-1] < Sq:
        L = min(int(torch.randint(lo, hi + 1, (1,), generator=gen).item()), Sq - cu_q[-1])
        P = int(torch.randint(0, prefix_hi + 1, (1,), generator=gen).item())
        if cu_k[-1] + P + L > Sk:
            break
        cu_q.append(cu_q[-1] + L)
        cu_k.append(cu_k[-1] + P + L)
    return torch.tensor(cu_q, dtype=torch.int32), torch.tensor(cu_k, dtype=torch.int32)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """CPU tensors for one workload: q, k, v, dO in the workload dtype; bias (workload dtype,
    [1|B, 1|Hq, Sq, Sk] per bias_dims) or None; sink fp32 [Hq] or None; seg int32 [B,S] or None; cu_q / cu_k
    int32 boundaries or None (thd_prefix workloads)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype

    def draw(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dt)

    q = draw((w.B, w.Sq, w.Hq, w.D), w.q_std)
    k = draw((w.B, w.Sk, w.Hkv, w.D), w.q_std)
    v = draw((w.B, w.Sk, w.Hkv, w.D), w.v_std)
    dO = draw((w.B, w.Sq, w.Hq, w.D), w.v_std)
    bias = None
    if w.bias:
        bias = draw(("b" in w.bias_dims and w.B or 1, "h" in w.bias_dims and w.Hq or 1, w.Sq, w.Sk), 1.0)
    sink = (torch.randn((w.Hq,), generator=g, dtype=torch.float32) * 5.0) if w.sink else None
    seg = None
    if w.segments:
        assert w.Sq == w.Sk
        seg = segment_runs(g, w.B, w.Sq, w.run_lo, w.run_hi)
    cu_q = cu_k = None
    if w.thd_prefix:
        assert w.B == 1
        cu_q, cu_k = thd_prefix_bounds(g, w.Sq, w.Sk, w.run_lo, w.run_hi, w.prefix_hi)
    return {"q": q, "k": k, "v": v, "dO": dO, "bias": bias, "sink": sink, "seg": seg, "cu_q": cu_q, "cu_k": cu_k}
