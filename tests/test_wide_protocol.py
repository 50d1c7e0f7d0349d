"""Model checks of the head-dim 320-512 (wide form) mbarrier protocols, run on the CPU with the
engine of test_bwd_protocol (random interleavings of the agents; a wait for phase k must see
k or k + 1 completed phases; deadlock is a failure).  MMAs complete at once (a commit is an
arrival).  Three kernels:

* the wide forward (fwd_tc.cu, wide form): one producer lane fills a single ring of two slots
  with the K slots of tile j and then the V slots of tile j - 1 (this CTA's part of O), in the
  MMA warp's order; S_j goes into score buffer j & 1, PV_{j-1} reads P_{j-1} there; two softmax
  agents (the two halves of a row), with the pair barrier and O rescaling of the tracked form.
  Data hazards: S_j may not overwrite P_{j-2} before PV_{j-2} has been issued and both halves
  have finished step j - 2; O may be rescaled at step j only with exactly j PVs completed.
* the wide backward's scores kernel (bwd_wide.cu): Q resident, K slots of every tile through a
  four-slot ring, then dO in Q's place (after every S MMA has read Q) and V slots; S / dP of
  tile jj into buffer jj & 1 once the element-wise warps have copied out tile jj - 2.
* the wide backward's GEMM kernel: a four-stage ring of A / B tiles and one accumulator
  barrier for the epilogue.

Each has a negative control with one wait removed, which the model must flag.
"""
import random
from collections import defaultdict

import pytest

from test_bwd_protocol import run_agents


def _counter(need):
    count, done = defaultdict(int), defaultdict(int)

    def arrive(b):
        count[b] += 1
        if count[b] == need[b]:
            count[b] = 0
            done[b] += 1

    return arrive, done


def simulate_wide_forward(n, nch, vh, fixm, rng, skip_p_wait=False):
    """n key tiles; nch 64-column chunks of the head dim; vh which CTA of the pair (its part of
    O: ceil(nch / 2) chunks for the first, floor(nch / 2) for the second); fixm: the fixed
    exponent offset (no pair barrier, no rescaling)."""
    NK = 2
    k_slots = (nch + 1) // 2
    vcn = (nch + 1) // 2 if vh == 0 else nch // 2
    v_slots = (vcn + 1) // 2
    need = defaultdict(lambda: 1)
    need.update({"p_full0": 2, "p_full1": 2})
    for j in range(n + 1):
        need[f"pair{j}"] = 2
    arrive, done = _counter(need)
    hazards = []
    state = {"pv": 0}

    def slot_waits(u):
        s = u % NK
        if u >= NK:
            yield ("wait", f"k_empty{s}", u // NK - 1)
        yield ("arrive", f"k_full{s}")

    def producer():
        yield ("arrive", "q_full")
        u = 0
        for j in range(n + 1):
            if j < n:
                for _ in range(k_slots):
                    yield from slot_waits(u)
                    u += 1
            if j >= 1:
                for _ in range(v_slots):
                    yield from slot_waits(u)
                    u += 1

    def mma():
        yield ("wait", "q_full", 0)
        u = 0
        for j in range(n + 1):
            if j < n:
                x = j & 1
                if j >= 2 and (done[f"p_full{x}"] < (j >> 1) or state["pv"] < j - 1):
                    hazards.append(("mma", f"S{j} over P{j - 2}", done[f"p_full{x}"], state["pv"]))
                for _ in range(k_slots):
                    s = u % NK
                    yield ("wait", f"k_full{s}", u // NK)
                    yield ("arrive", f"k_empty{s}")
                    u += 1
                yield ("arrive", f"s_full{x}")
            if j >= 1:
                jj = j - 1
                if not skip_p_wait:
                    yield ("wait", f"p_full{jj & 1}", jj >> 1)
                if done[f"p_full{jj & 1}"] < (jj >> 1) + 1:
                    hazards.append(("mma", f"PV{jj} before P{jj}", done[f"p_full{jj & 1}"]))
                for _ in range(v_slots):
                    s = u % NK
                    yield ("wait", f"k_full{s}", u // NK)
                    yield ("arrive", f"k_empty{s}")
                    u += 1
                state["pv"] += 1
                yield ("arrive", "o_done")
        if fixm:
            yield ("arrive", "o_fin")

    def softmax(half):
        for j in range(n):
            yield ("wait", f"s_full{j & 1}", j >> 1)
            if not fixm:
                yield ("arrive", f"pair{j}")
                yield ("wait", f"pair{j}", 0)
                if j >= 1:
                    yield ("wait", "o_done", j - 1)
                    if state["pv"] != j:
                        hazards.append((f"softmax{half}", f"rescale O at {j}", state["pv"]))
            yield ("arrive", f"p_full{j & 1}")
        if n > 0:
            yield ("wait", "o_fin", 0) if fixm else ("wait", "o_done", n - 1)

    agents = {"producer": producer(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)}
    return run_agents(agents, arrive, done, hazards, rng)


def simulate_wide_scores(n, nch, rng, skip_free_wait=False):
    """The scores kernel for n key tiles and nch head-dim chunks: 2 n score tiles (S_0..S_{n-1},
    then dP_0..dP_{n-1}) through two TMEM buffers."""
    NR = 4
    need = defaultdict(lambda: 1)
    need.update({"p_free0": 2, "p_free1": 2})
    arrive, done = _counter(need)
    hazards = []
    state = {"s_issued": 0}

    def slot(u):
        s = u % NR
        if u >= NR:
            yield ("wait", f"r_empty{s}", u // NR - 1)
        yield ("arrive", f"r_full{s}")

    def producer():
        yield ("arrive", "q_full")
        u = 0
        for _ in range(n):
            for _ in range(nch):
                yield from slot(u)
                u += 1
        yield ("wait", "q_free", 0)
        if state["s_issued"] < n:
            hazards.append(("producer", "dO over Q before every S", state["s_issued"]))
        yield ("arrive", "do_full")
        for _ in range(n):
            for _ in range(nch):
                yield from slot(u)
                u += 1

    def mma():
        yield ("wait", "q_full", 0)
        u = 0
        for jj in range(2 * n):
            if jj == n:
                yield ("wait", "do_full", 0)
            x = jj & 1
            if jj >= 2:
                if not skip_free_wait:
                    yield ("wait", f"p_free{x}", (jj - 2) >> 1)
                if done[f"p_free{x}"] < ((jj - 2) >> 1) + 1:
                    hazards.append(("mma", f"tile {jj} over tile {jj - 2}", done[f"p_free{x}"]))
            for _ in range(nch):
                s = u % NR
                yield ("wait", f"r_full{s}", u // NR)
                yield ("arrive", f"r_empty{s}")
                u += 1
            yield ("arrive", f"s_full{x}")
            if jj < n:
                state["s_issued"] += 1
            if jj == n - 1:
                yield ("arrive", "q_free")

    def elementwise():
        for jj in range(2 * n):
            yield ("wait", f"s_full{jj & 1}", jj >> 1)
            yield ("arrive", f"p_free{jj & 1}")

    agents = {"producer": producer(), "mma": mma(), "ew0": elementwise(), "ew1": elementwise()}
    return run_agents(agents, arrive, done, hazards, rng)


def simulate_wide_gemm(total, rng, skip_empty_wait=False):
    """The GEMM kernel with `total` contraction steps through a four-stage ring."""
    ST = 4
    need = defaultdict(lambda: 1)
    arrive, done = _counter(need)
    hazards = []
    consumed = defaultdict(int)

    def producer():
        for it in range(total):
            s = it % ST
            if it >= ST and not skip_empty_wait:
                yield ("wait", f"f_empty{s}", it // ST - 1)
            if consumed[s] < it // ST:
                hazards.append(("producer", f"stage {s} refilled before use {it // ST - 1} was read", consumed[s]))
            yield ("arrive", f"f_full{s}")

    def mma():
        for it in range(total):
            s = it % ST
            yield ("wait", f"f_full{s}", it // ST)
            consumed[s] += 1
            yield ("arrive", f"f_empty{s}")
        yield ("arrive", "acc_full")

    def epilogue():
        if total > 0:
            yield ("wait", "acc_full", 0)
            if sum(consumed.values()) != total:
                hazards.append(("epilogue", "accumulator read early", sum(consumed.values())))

    agents = {"producer": producer(), "mma": mma(), "epilogue": epilogue()}
    return run_agents(agents, arrive, done, hazards, rng)


@pytest.mark.parametrize("nch", [5, 6, 7, 8])
@pytest.mark.parametrize("fixm", [True, False])
def test_wide_forward_protocol(nch, fixm):
    rng = random.Random(7 * nch + int(fixm))
    for n in [1, 2, 3, 4, 5, 9]:
        for vh in (0, 1):
            for _ in range(60):
                ok, hz = simulate_wide_forward(n, nch, vh, fixm, rng)
                assert ok, ("deadlock", n, nch, vh, fixm)
                assert not hz, (n, nch, vh, fixm, hz[:3])


def test_wide_forward_model_flags_pv_without_its_wait():
    rng = random.Random(3)
    flagged = 0
    for _ in range(200):
        ok, hz = simulate_wide_forward(4, 8, 0, True, rng, skip_p_wait=True)
        flagged += bool(hz) or not ok
    assert flagged > 0


@pytest.mark.parametrize("nch", [5, 6, 7, 8])
def test_wide_scores_protocol(nch):
    rng = random.Random(11 * nch)
    for n in [1, 2, 3, 4]:
        for _ in range(80):
            ok, hz = simulate_wide_scores(n, nch, rng)
            assert ok, ("deadlock", n, nch)
            assert not hz, (n, nch, hz[:3])


def test_wide_scores_model_flags_missing_free_wait():
    rng = random.Random(5)
    flagged = 0
    for _ in range(200):
        ok, hz = simulate_wide_scores(3, 8, rng, skip_free_wait=True)
        flagged += bool(hz) or not ok
    assert flagged > 0


def test_wide_gemm_protocol_and_its_negative_control():
    rng = random.Random(13)
    for total in [0, 1, 3, 4, 5, 9, 17]:
        for _ in range(80):
            ok, hz = simulate_wide_gemm(total, rng)
            assert ok and not hz, (total, hz[:3])
    flagged = 0
    for _ in range(200):
        ok, hz = simulate_wide_gemm(9, rng, skip_empty_wait=True)
        flagged += bool(hz) or not ok
    assert flagged > 0
