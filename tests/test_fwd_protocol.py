"""Model check of the tensor-core forward's mbarrier protocol (attention_flash_attn_gb300/csrc/
fwd_tc.cu), run on the CPU with the engine of test_bwd_protocol.

Agents: the K loader (TMA lane 0), the V loader (lane 1), the MMA warp (S_j into score buffer
j & 1, then PV_{j-1} reading P_{j-1} from TMEM), and the two softmax warps of a lane quarter
(one agent per half row; they meet at a pair barrier in the tracked-maximum form).  MMAs
complete at once (a commit is an arrival).  Besides deadlock and the parity rule (a wait for
phase k must see k or k + 1 completed phases), two data hazards are checked:

* S_{j+2} reuses the score buffer of S_j and P_j: the MMA warp may issue it only after both
  softmax warps have finished step j (arrived on p_full for it);
* the tracked-maximum form rescales O in TMEM at step j: no PV may be in flight then, so
  exactly j PVs have completed;
* each softmax warp writes P_j over score columns: in the kernel's layout a warp writes only
  into its own half of S_j; in the earlier layout the second half's P went over columns of
  the first half's S, which the fixed-offset form (no pair barrier per step) does not order
  after the first half's reads -- the negative control.

Ring shapes: head dim 64 (4 K / 4 V stages), 128 (3 / 2), 256 (one K and one V tile, each
filled and released in two halves with barriers of their own).
"""
import random
from collections import defaultdict

import pytest

from test_bwd_protocol import run_agents

TILE_COUNTS = [1, 2, 3, 4, 5, 7, 9, 16, 33]


def simulate_forward(n, nk, nv, halves, fixm, rng, skip_pv_wait=False, p_layout="own"):
    """Returns (finished, hazards).  halves: the head-dim-256 form (K by head-dim halves, V by
    key halves, each half its own full / empty barrier pair).  skip_pv_wait drops the MMA
    warp's wait on p_full before PV (a negative control: P would be read before it is
    written and the buffer overwritten early)."""
    need = defaultdict(lambda: 1)
    need.update({"p_full0": 2, "p_full1": 2})
    for j in range(n + 1):
        need[f"pair{j}"] = 2
    count, done, hazards = defaultdict(int), defaultdict(int), []

    def arrive(b):
        count[b] += 1
        if count[b] == need[b]:
            count[b] = 0
            done[b] += 1

    def ring_loader(kind, depth):
        for j in range(n):
            if halves:
                for hf in range(2):
                    if j >= 1:
                        yield ("wait", f"{kind}_empty{hf}", j - 1)
                    yield ("arrive", f"{kind}_full{hf}")
            else:
                s = j % depth
                if j >= depth:
                    yield ("wait", f"{kind}_empty{s}", j // depth - 1)
                yield ("arrive", f"{kind}_full{s}")

    def kload():
        yield ("arrive", "q_full")
        yield from ring_loader("k", nk)

    def mma():
        yield ("wait", "q_full", 0)
        for j in range(n + 1):
            if j < n:
                x = j & 1
                if halves:
                    for hf in range(2):
                        yield ("wait", f"k_full{hf}", j)
                        yield ("arrive", f"k_empty{hf}")
                else:
                    yield ("wait", f"k_full{j % nk}", j // nk)
                if j >= 2 and done[f"p_full{x}"] < (j >> 1):
                    hazards.append(("mma", f"S{j} over P{j - 2}", j, done[f"p_full{x}"]))
                yield ("arrive", f"s_full{x}")
                if not halves:
                    yield ("arrive", f"k_empty{j % nk}")
            if j >= 1:
                jj = j - 1
                if halves:
                    if not skip_pv_wait:
                        yield ("wait", f"p_full{jj & 1}", jj >> 1)
                    for hf in range(2):
                        yield ("wait", f"v_full{hf}", jj)
                        yield ("arrive", f"v_empty{hf}")
                else:
                    yield ("wait", f"v_full{jj % nv}", jj // nv)
                    if not skip_pv_wait:
                        yield ("wait", f"p_full{jj & 1}", jj >> 1)
                    yield ("arrive", f"v_empty{jj % nv}")
                yield ("arrive", "o_done")
        if fixm:
            yield ("arrive", "o_fin")

    def softmax(half):
        for j in range(n):
            yield ("wait", f"s_full{j & 1}", j >> 1)
            yield ("arrive", f"sread{half}")  # this half's S_j is in registers
            if not fixm:
                yield ("arrive", f"pair{j}")  # exchange of half-row maxima
                yield ("wait", f"pair{j}", 0)
                if j >= 1:
                    yield ("wait", "o_done", j - 1)
                    if done["o_done"] != j:
                        hazards.append(("softmax", "O rescaled under a PV", j, done["o_done"]))
            if p_layout == "shared" and half == 1 and done["sread0"] <= j:
                hazards.append(("softmax1", "P over the partner's S", j, done["sread0"]))
            yield ("arrive", f"p_full{j & 1}")
        if n > 0:
            if fixm:
                yield ("wait", "o_fin", 0)
            else:
                yield ("wait", "o_done", n - 1)
        yield ("arrive", f"pair{n}")  # the row sums are combined
        yield ("wait", f"pair{n}", 0)

    agents = {"kload": kload(), "vload": ring_loader("v", nv), "mma": mma(),
              "softmax0": softmax(0), "softmax1": softmax(1)}
    return run_agents(agents, arrive, done, hazards, rng)


SHAPES = [(4, 4, False), (3, 2, False), (1, 1, True)]


@pytest.mark.parametrize("nk,nv,halves", SHAPES, ids=["d64", "d128", "d256"])
@pytest.mark.parametrize("fixm", [False, True], ids=["tracked", "fixed"])
def test_forward_protocol_never_deadlocks_aliases_or_races(nk, nv, halves, fixm):
    rng = random.Random(nk * 10 + nv + (100 if fixm else 0))
    for trial in range(400):
        n = TILE_COUNTS[trial % len(TILE_COUNTS)]
        finished, hazards = simulate_forward(n, nk, nv, halves, fixm, rng)
        assert finished and not hazards, (n, hazards[:3])


@pytest.mark.parametrize("fixm", [False, True], ids=["tracked", "fixed"])
def test_forward_model_flags_pv_without_the_p_full_wait(fixm):
    """Negative control: with PV issued before the softmax has written P, the next S MMA
    overwrites a score buffer that still holds P (and barrier phases alias)."""
    rng = random.Random(9)
    over_p = 0
    for trial in range(200):
        _, hazards = simulate_forward(8, 4, 4, False, fixm, rng, skip_pv_wait=True)
        over_p += sum(1 for h in hazards if " over P" in h[1])
    assert over_p > 0


def test_forward_model_flags_p_over_the_partner_s_without_a_pair_barrier():
    """Negative control: with the second half's P written over the first half's score columns,
    the fixed-offset form (no per-step pair barrier) lets the write overtake the partner's
    read; the tracked form's pair barrier orders them."""
    rng = random.Random(17)
    flagged = {True: 0, False: 0}
    for fixm in (True, False):
        for trial in range(200):
            _, hazards = simulate_forward(8, 1, 1, True, fixm, rng, p_layout="shared")
            flagged[fixm] += sum(1 for h in hazards if "partner" in h[1])
    assert flagged[True] > 0 and flagged[False] == 0
