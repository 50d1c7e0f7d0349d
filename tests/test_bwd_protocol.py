"""Model check of the tensor-core backward's mbarrier protocols (attention_flash_attn_gb300/
csrc/bwd_tc.cu), run on the CPU: the head-dim-256 two-pass form and the one-pass form.

Each agent of the kernel -- TMA lanes 0 and 1, the front MMA warp (S^T, dK, dP^T), the
back MMA warp (dV, dQ), the softmax warps, the dQ drain -- is a generator that yields the
waits and arrivals it performs, in program order.  MMAs complete at once (a commit is an
arrival).  Waits use the hardware's parity rule: a wait for phase k of a barrier returns
when the barrier's completed-phase count has the other parity, so it is only sound if the
count is k or k + 1 when the waiter looks.  Random schedules must always finish, and no
waiter may ever see a count outside {k, k + 1}.

simulate_split_rings is the two-pass form's protocol (two Q slots and one dO slot in the dK
pass, double-buffered dS^T with one ready barrier per buffer).  Its negative control hands
both dS^T buffers over through a single ready barrier: the softmax can then complete two
phases ahead of the back MMA warp, which the model must flag.  simulate_fused is the one-pass
form (head dims 64 and 128), with the front warp's MMAs completing asynchronously, so that it
can also check that no stage is refilled while they still read it; its negative control drops
the s_full chain.
"""
import random
from collections import defaultdict


STEP_COUNTS = [1, 2, 3, 4, 5, 6, 8, 13, 33, 66, 80]


def run_agents(agents, arrive, done, hazards, rng):
    pending = dict.fromkeys(agents)
    finished = set()
    while len(finished) < len(agents):
        progress = False
        turn = list(agents)
        rng.shuffle(turn)
        for name in turn:
            if name in finished:
                continue
            for _ in range(rng.randint(1, 8)):
                op = pending[name]
                if op is None:
                    try:
                        op = pending[name] = next(agents[name])
                    except StopIteration:
                        finished.add(name)
                        progress = True
                        break
                if op[0] == "arrive":
                    arrive(op[1])
                    pending[name] = None
                    progress = True
                    continue
                _, bar, phase = op
                if done[bar] not in (phase, phase + 1):
                    hazards.append((name, bar, phase, done[bar]))
                if (done[bar] & 1) != (phase & 1):
                    pending[name] = None
                    progress = True
                else:
                    break
        if not progress:
            return False, hazards
    return True, hazards


def simulate_split_rings(nper, rng, single_ready=False):
    """The head-dim-256 protocol: K resident; dV pass over two Q / dO stages; then V in tensor
    memory, the dK pass's tiles in two rings (two Q slots, one dO slot), S^T and dP^T sharing
    one score buffer, dQ^T drained one 128-row half at a time, and dS double-buffered: each dS
    buffer has its own ready barrier and its own MMA-completion barrier (dK + dQ of the step
    that read it), so the softmax never waits on the step it has just handed over.
    single_ready: the dK pass's dS buffers share one ready barrier (negative control).
    Returns (finished, hazards)."""
    prb = (lambda i: "p_ready") if single_ready else (lambda i: f"prb{i & 1}")
    prb_phase = (lambda i: nper + i) if single_ready else (lambda i: i >> 1)
    nsteps, nB = 2 * nper, nper
    need = defaultdict(lambda: 1)
    need.update({"mma_done": 2, "mdb0": 2, "mdb1": 2, "fin_done": 2})  # p_ready etc.: one arrival (the model's softmax is one agent)
    count, done, hazards = defaultdict(int), defaultdict(int), []

    def arrive(b):
        count[b] += 1
        if count[b] == need[b]:
            count[b] = 0
            done[b] += 1

    u_last0, u_last1 = ((nper + 1) >> 1) - 1, (nper >> 1) - 1

    def loader0():
        yield ("arrive", "kv_full")
        for j in range(nsteps):
            if j >= 2:
                yield ("wait", f"ld_empty{j & 1}", (j >> 1) - 1)
            yield ("arrive", f"ld_full{j & 1}")
            if j < nper:
                s, u = j & 1, j >> 1
                if u >= 1:
                    yield ("wait", f"qdo_empty{s}", u - 1)
                yield ("arrive", f"qdo_full{s}")
                continue
            i = j - nper
            r = i & 1  # Q_i
            if i >= 2:
                yield ("wait", f"ring_empty{r}", (i >> 1) - 1)
            elif r == 0:
                yield ("wait", "qdo_empty0", u_last0)
            else:
                yield ("wait", "do0_free", 0)
            yield ("arrive", f"ring_full{r}")
            if i >= 1:  # dO_i
                yield ("wait", "ring_empty2", i - 1)
            elif u_last1 >= 0:
                yield ("wait", "qdo_empty1", u_last1)
            yield ("arrive", "ring_full2")

    def loader1():
        for j in range(nper):
            s, u = j & 1, j >> 1
            if u >= 1:
                yield ("wait", f"do_empty{s}", u - 1)
            yield ("arrive", f"do_full{s}")
        if nper > 0:
            yield ("wait", "do_empty0", u_last0)
            yield ("arrive", "do0_free")

    def front():
        yield ("wait", "kv_full", 0)
        for j in range(nper):
            if j >= 1:
                yield ("wait", "sdp_free", j - 1)
            yield ("wait", f"qdo_full{j & 1}", j >> 1)
            yield ("arrive", "s_full")
            yield ("arrive", f"qdo_empty{j & 1}")

        def dk(i):
            yield ("wait", prb(i), prb_phase(i))
            yield ("arrive", f"ring_empty{i & 1}")
            yield ("arrive", f"mdb{i & 1}")

        for i in range(nB):
            j = nper + i
            if i == 0:
                yield ("wait", "sdp_free", nper - 1)
                yield ("wait", "acc_free", 0)
            else:
                yield ("wait", "dp_free", i - 1)
            yield ("wait", f"ring_full{i & 1}", i >> 1)
            yield ("arrive", "s_full")
            if i >= 1:
                yield from dk(i - 1)
            yield ("wait", "sdp_free", j)
            if i == 0:
                yield ("wait", "v_full", 0)
            yield ("wait", "ring_full2", i)
            yield ("arrive", "ring_empty2")
            yield ("arrive", "dp_full")
        if nB > 0:
            yield from dk(nB - 1)
        yield ("arrive", "fin_done")

    def back():
        yield ("wait", "kv_full", 0)
        h = 0
        for j in range(1, nsteps + 1):
            jj = j - 1
            if jj < nper:
                yield ("wait", "p_ready", jj)
                yield ("wait", f"do_full{jj & 1}", jj >> 1)
                yield ("arrive", f"do_empty{jj & 1}")
                yield ("arrive", "mma_done")
                yield ("arrive", "mma_done")
                continue
            yield ("wait", prb(jj - nper), prb_phase(jj - nper))
            for _ in range(2):
                if h >= 1:
                    yield ("wait", "dq_empty", h - 1)
                yield ("arrive", "dq_full")
                h += 1
            yield ("arrive", f"mdb{(jj - nper) & 1}")
        yield ("arrive", "fin_done")

    def softmax():
        for j in range(nsteps):
            yield ("wait", "s_full", j)
            yield ("wait", f"ld_full{j & 1}", j >> 1)
            yield ("arrive", "sdp_free")
            if j >= nper:
                yield ("wait", "dp_full", j - nper)
                yield ("arrive", "dp_free")
            yield ("arrive", f"ld_empty{j & 1}")
            if j < nper:
                if j >= 1:
                    yield ("wait", "mma_done", j - 1)
            else:
                i = j - nper
                if i >= 2:  # dS buffer i & 1 was last read by dK / dQ of step i - 2
                    yield ("wait", f"mdb{i & 1}", (i >> 1) - 1)
            # dV pass: one p_ready; dK pass: one per dS buffer, so that its phases are two
            # steps apart and the MMA warps cannot be overtaken twice
            yield ("arrive", "p_ready" if j < nper else prb(j - nper))
            if j == nper - 1:
                yield ("wait", "mma_done", j)
                yield ("arrive", "acc_free")
                yield ("arrive", "v_full")
        if nsteps > 0:
            yield ("wait", "fin_done", 0)

    def drain():
        for h in range(2 * nB):
            yield ("wait", "dq_full", h)
            yield ("arrive", "dq_empty")

    return run_agents({"loader0": loader0(), "loader1": loader1(), "front": front(), "back": back(),
                       "softmax": softmax(), "drain": drain()}, arrive, done, hazards, rng)


def test_split_rings_protocol_never_deadlocks_or_aliases():
    rng = random.Random(777)
    for trial in range(1500):
        nper = STEP_COUNTS[trial % len(STEP_COUNTS)]
        finished, hazards = simulate_split_rings(nper, rng)
        assert finished and not hazards, (nper, hazards[:3])


def test_split_rings_model_flags_a_single_ready_barrier():
    """Negative control: with one ready barrier for both dS^T buffers, the softmax can arrive
    for two dK-pass steps before the back warp looks for the first, a phase the parity wait
    cannot tell from the one two later."""
    rng = random.Random(99)
    flagged = 0
    for trial in range(400):
        finished, hazards = simulate_split_rings(13, rng, single_ready=True)
        flagged += (not finished) or bool(hazards)
    assert flagged > 0


def simulate_fused(nsteps, rng, ns=3, skip_chain=False):
    """The one-pass form (head dims 64 and 128): a ring of ns Q / dO stages (each also holding
    the step's LSE and -D tile), filled by the TMA lane and released by the back MMA warp's
    commit; the front warp issues S^T, the K = 16 MMA that starts dP^T at -D, and dP^T; the
    back warp dV, dK, dQ.  The front warp's commit does not cover the stage's release, so the
    -D tile (read by the front warp's init MMA) may only be refilled once s_full of its step
    has completed: the model's loader refills a stage on qdo_empty, which the back warp commits
    only after p_ready, which the softmax arrives on only after s_full.  skip_chain drops the
    softmax's wait on s_full (so nothing orders the refill after the front warp's MMAs) and the
    model must then report the refill racing the init MMA."""
    need = defaultdict(lambda: 1)
    need.update({"fin_done": 2})  # front and back MMA warps
    count, done, hazards = defaultdict(int), defaultdict(int), []
    reads = defaultdict(int)  # stage -> front-warp MMAs issued on it and not yet complete

    def arrive(b):
        count[b] += 1
        if count[b] == need[b]:
            count[b] = 0
            done[b] += 1

    slot, use = (lambda j: j % ns), (lambda j: j // ns)

    def loader():
        yield ("arrive", "kv_full")
        for j in range(nsteps):
            s, u = slot(j), use(j)
            if u >= 1:
                yield ("wait", f"qdo_empty{s}", u - 1)
                if reads[s]:
                    hazards.append(("loader", f"stage{s}", u, "refilled under the init MMA"))
            yield ("arrive", f"qdo_full{s}")

    def front():
        yield ("wait", "kv_full", 0)
        for j in range(nsteps):
            if j >= 1:
                yield ("wait", "sdp_free", j - 1)
            yield ("wait", f"qdo_full{slot(j)}", use(j))
            reads[slot(j)] += 1  # S^T, the -D init and dP^T read the stage
            yield ("arrive", f"issued{j}")  # handed to the tensor pipe; completes later
        yield ("arrive", "fin_done")

    def tensor_pipe():  # completes the front warp's MMAs in issue order, then its commit arrives
        for j in range(nsteps):
            yield ("wait", f"issued{j}", 0)
            reads[slot(j)] -= 1
            yield ("arrive", "s_full")

    def back():
        yield ("wait", "kv_full", 0)
        for j in range(1, nsteps + 1):
            jj = j - 1
            yield ("wait", "p_ready", jj)
            if jj >= 1:
                yield ("wait", "dq_empty", jj - 1)
            yield ("arrive", "dq_full")
            yield ("arrive", "mma_done")
            yield ("arrive", f"qdo_empty{slot(jj)}")
        yield ("arrive", "fin_done")

    def softmax():
        for j in range(nsteps):
            if not skip_chain:
                yield ("wait", "s_full", j)
            yield ("wait", f"qdo_full{slot(j)}", use(j))
            yield ("arrive", "sdp_free")
            if j >= 1:
                yield ("wait", "mma_done", j - 1)
            yield ("arrive", "p_ready")
        if nsteps > 0:
            yield ("wait", "fin_done", 0)

    def drain():
        for h in range(nsteps):
            yield ("wait", "dq_full", h)
            yield ("arrive", "dq_empty")

    return run_agents({"loader": loader(), "front": front(), "tensor": tensor_pipe(), "back": back(),
                       "softmax": softmax(), "drain": drain()}, arrive, done, hazards, rng)


def test_fused_protocol_never_deadlocks_aliases_or_refills_under_the_init_mma():
    rng = random.Random(4242)
    for trial in range(1500):
        nsteps = STEP_COUNTS[trial % len(STEP_COUNTS)]
        finished, hazards = simulate_fused(nsteps, rng)
        assert finished and not hazards, (nsteps, hazards[:3])


def test_fused_model_flags_a_refill_without_the_s_full_chain():
    rng = random.Random(5)
    flagged = False
    for trial in range(300):
        finished, hazards = simulate_fused(12, rng, skip_chain=True)
        flagged |= any(h[3] == "refilled under the init MMA" for h in hazards if len(h) == 4)
    assert flagged
