"""Pins for the fp64 oracle: each test fixes part of it against something other than itself
(finite differences, a library routine, closed forms, invariants, brute force).

A plausible slip anywhere in the oracle -- a dropped term, a wrong sign or index, a
transposed operand, the cap or bias in the wrong place, the sink counted twice --
fails at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import Problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")
FIG = json.load(open(GOLDEN))


def rng(seed=0):
    return np.random.default_rng(seed)


def full_problem(S=7, D=4, Hq=2, Hkv=1, B=1, seed=0, cap=2.0, causal=True, window=4,
                 bias=True, sink=True, segs=True, q_std=1.5, Sk=None):
    Sk = S if Sk is None else Sk
    r = rng(seed)
    q = r.normal(0, q_std, (B, S, Hq, D))
    k = r.normal(0, q_std, (B, Sk, Hkv, D))
    v = r.normal(0, 1, (B, Sk, Hkv, D))
    kw = dict(scale=1 / math.sqrt(D), causal=causal, window=window, softcap=cap)
    if bias:
        kw["bias"] = r.normal(0, 1, (1, Hq, S, Sk))
    if sink:
        kw["sink"] = r.normal(0, 1, (Hq,))
    if segs:
        # the last query and the last key share the second segment (bottom-right alignment)
        seg_q = np.zeros((B, S), np.int32)
        seg_q[:, S // 2 + 1:] = 1
        seg_k = np.zeros((B, Sk), np.int32)
        seg_k[:, Sk - (S - S // 2 - 1):] = 1
        kw["seg_q"], kw["seg_k"] = seg_q, seg_k
    return Problem(q, k, v, **kw), r.normal(0, 1, (B, S, Hq, D))


def loss(p, dO):
    O, _ = oracle.forward(p)
    return float(np.sum(O * dO))


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ----------------------------------------------------------------- whole fwd / bwd

@pytest.mark.parametrize("S,Sk,causal", [(5, 5, True), (7, 7, True), (5, 8, True), (5, 8, False),
                                         (8, 5, True)])
def test_backward_matches_central_finite_differences(S, Sk, causal):
    """Analytic dQ, dK, dV, dbias, dsink equal central differences of sum(O*dO) in fp64
    (bias + sink + cap + window + segments all on, causal or not), also with fewer queries
    than keys and more queries than keys, where the window is measured from each query's
    bottom-right aligned position."""
    p, dO = full_problem(S=S, Sk=Sk, causal=causal, window=3 if Sk != S else 4)
    O, LSE = oracle.forward(p)
    g = oracle.backward(p, dO, O, LSE)
    h = 1e-5

    def fd(name):
        base = getattr(p, name)
        out = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = base[idx]
            base[idx] = orig + h
            lp = loss(p, dO)
            base[idx] = orig - h
            lm = loss(p, dO)
            base[idx] = orig
            out[idx] = (lp - lm) / (2 * h)
        return out

    for name, key in [("q", "dq"), ("k", "dk"), ("v", "dv"), ("bias", "dbias"), ("sink", "dsink")]:
        num = fd(name)
        assert rel(g[key], num) <= 1e-6, (name, rel(g[key], num))


# ----------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_vanilla_equals_torch_sdpa_fp64(causal, with_bias):
    """cap = 0, no sink/window/segments: the oracle equals torch's scaled_dot_product_attention
    in fp64 on the CPU, and its gradients equal autograd's (bias = additive float mask)."""
    r = rng(1)
    B, S, H, D = 2, 19, 3, 8
    q, k, v, dO = (r.normal(0, 1, (B, S, H, D)) for _ in range(4))
    bias = r.normal(0, 1, (B, H, S, S)) if with_bias else None
    p = Problem(q, k, v, scale=1 / math.sqrt(D), causal=causal, bias=bias)
    O, LSE = oracle.forward(p)
    g = oracle.backward(p, dO, O, LSE)

    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
    mask = None
    tb = None
    if with_bias:
        tb = torch.tensor(bias, requires_grad=True)
        mask = tb
        if causal:
            keep = torch.ones(S, S, dtype=torch.bool).tril()
            mask = tb.masked_fill(~keep, float("-inf"))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask, is_causal=causal and not with_bias, scale=1 / math.sqrt(D))
    ref.backward(torch.tensor(dO.transpose(0, 2, 1, 3)))
    assert rel(O, ref.detach().numpy().transpose(0, 2, 1, 3)) <= 1e-12
    assert rel(g["dq"], tq.grad.numpy().transpose(0, 2, 1, 3)) <= 1e-12
    assert rel(g["dk"], tk.grad.numpy().transpose(0, 2, 1, 3)) <= 1e-12
    assert rel(g["dv"], tv.grad.numpy().transpose(0, 2, 1, 3)) <= 1e-12
    if with_bias:
        assert rel(g["dbias"], tb.grad.numpy()) <= 1e-12


def test_lse_equals_torch_logsumexp():
    """LSE is the natural log of the softmax normaliser (sink included as one more column)."""
    r = rng(2)
    B, S, H, D = 1, 11, 2, 4
    q, k, v = (r.normal(0, 1, (B, S, H, D)) for _ in range(3))
    sink = r.normal(0, 3, (H,))
    p = Problem(q, k, v, scale=0.5, sink=sink)
    _, LSE = oracle.forward(p)
    logits = torch.einsum("bihd,bjhd->bhij", torch.tensor(q), torch.tensor(k)) * 0.5
    cols = torch.cat([logits, torch.tensor(sink).view(1, H, 1, 1).expand(B, H, S, 1)], dim=-1)
    assert rel(LSE, torch.logsumexp(cols, dim=-1).numpy()) <= 1e-14


# ----------------------------------------------------------------- the cap

def test_softcap_closed_forms():
    """cap*tanh(u/cap): odd, below cap, exact at u = cap*atanh(1/2), cubic Taylor term,
    saturating at +-cap, and identity when off."""
    for cap in (1.0, 30.0, 50.0):
        p = Problem(np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)),
                    scale=1.0, softcap=cap)
        assert oracle.capped(p, cap * math.atanh(0.5)) == pytest.approx(cap / 2, rel=1e-15)
        for u in (-200.0, -3.0, 0.7, 29.0, 168.0):
            t = oracle.capped(p, u)
            assert abs(t) <= cap and t == -oracle.capped(p, -u)
            if abs(u) / cap < 18:
                assert abs(t) < cap
        assert oracle.capped(p, 1e4) == cap and oracle.capped(p, -1e4) == -cap
    big = Problem(np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)),
                  scale=1.0, softcap=1e3)
    for u in (0.5, 3.0, 10.0):
        assert abs(oracle.capped(big, u) - (u - u ** 3 / (3 * 1e6))) <= 1e-7 * max(1, u ** 5 / 1e5)
    off = Problem(np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)), scale=1.0)
    assert oracle.capped(off, 123.5) == 123.5 and oracle.cap_factor(off, 123.5) == 1.0


def test_softcap_factor_is_derivative():
    """The backward factor equals d/du of the capped logit (central differences), including
    far in the saturated range where 1 - tanh^2 is tiny (u = 168, cap = 30)."""
    fig = FIG["softcap_active_range"]
    p = Problem(np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)), np.zeros((1, 1, 1, 1)),
                scale=1.0, softcap=fig["cap"])
    for u in (-fig["max_pre_cap_logit"], -40.0, -1.0, 0.0, 2.5, 31.0, 90.0):
        h = 1e-4
        num = (oracle.capped(p, u + h) - oracle.capped(p, u - h)) / (2 * h)
        assert oracle.cap_factor(p, u) == pytest.approx(num, rel=1e-6, abs=1e-12)


def test_cap_applies_after_bias_and_before_mask():
    """Two keys with q.k = 0: bias 100 on key 0, cap 1.  Capped after the bias add, key 0's
    logit is exactly 1 (tanh(100) == 1 in fp64), so O = sigmoid(1) v0 + sigmoid(-1) v1.
    A third key masked out by causality carries a huge bias and must not matter."""
    q = np.zeros((1, 3, 1, 2))
    k = np.zeros((1, 3, 1, 2))
    v = np.array([[[[1.0, 0.0]], [[0.0, 1.0]], [[7.0, 7.0]]]])
    bias = np.zeros((1, 1, 3, 3))
    bias[0, 0, 1, 0] = 100.0
    bias[0, 0, 1, 2] = 1e6        # masked (j = 2 > i = 1 under causal)
    p = Problem(q, k, v, scale=1.0, causal=True, softcap=1.0, bias=bias)
    O, _ = oracle.forward(p, rows=[1])
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(O[0, 1, 0], [s1, 1 - s1], rtol=1e-15)


def test_capped_logits_bounded_in_attention():
    """With the cap active, every visible logit is inside (-cap, cap): recovered as
    LSE_i - ln(number of visible keys) bounds on one-key rows (segments of length 1)."""
    r = rng(3)
    S, D, cap = 9, 4, 2.0
    q, k, v = r.normal(0, 10, (1, S, 1, D)), r.normal(0, 10, (1, S, 1, D)), r.normal(0, 1, (1, S, 1, D))
    seg = np.arange(S, dtype=np.int32)[None]          # every token its own segment
    p = Problem(q, k, v, scale=1.0, softcap=cap, seg_q=seg)
    _, LSE = oracle.forward(p)
    u = np.einsum("bihd,bihd->bhi", q, k)             # the one visible key of each row
    assert np.all(np.abs(LSE) <= cap)                 # one visible key: LSE == its capped logit
    assert np.all(np.abs(LSE[np.abs(u) < 18 * cap]) < cap)
    assert np.all(np.sign(LSE) == np.sign(u))
    assert np.max(np.abs(u)) > 18 * cap               # cap really active


# ----------------------------------------------------------------- normalisation and the sink

def test_probabilities_plus_sink_sum_to_one():
    """v_j = e_j (one-hot, D = Sk): O_i holds the row of P, so sum_j P_ij + p0_i = 1."""
    r = rng(4)
    S, Hq = 12, 2
    q = r.normal(0, 2, (1, S, Hq, S))
    k = r.normal(0, 2, (1, S, 1, S))
    v = np.eye(S)[None, :, None, :]
    sink = r.normal(0, 5, (Hq,))
    seg = np.array([[0] * 5 + [1] * 7], np.int32)
    p = Problem(q, k, v, scale=0.3, causal=True, window=6, softcap=3.0, sink=sink, seg_q=seg)
    O, LSE = oracle.forward(p)
    p0 = np.exp(sink[None, :, None] - LSE)            # [B,Hq,Sq]
    tot = O.sum(-1).transpose(0, 2, 1) + p0
    np.testing.assert_allclose(tot, 1.0, atol=1e-14)


@pytest.mark.parametrize("cap", [0.0, 4.0])
def test_sink_single_key_closed_form(cap):
    """One query, one key: O = sigmoid(t - s) v, LSE = ln(e^t + e^s),
    dsink = -p0 (dO.O), dv = sigmoid(t - s) dO."""
    a, b, s = 1.5, 2.0, 0.75
    q = np.array([[[[a, 0.0]]]])
    k = np.array([[[[b, 0.0]]]])
    v = np.array([[[[0.3, -1.2]]]])
    dO = np.array([[[[0.5, 2.0]]]])
    u = a * b                                          # scale 1
    t = cap * math.tanh(u / cap) if cap else u         # cap written out for this single value
    p = Problem(q, k, v, scale=1.0, softcap=cap, sink=np.array([s]))
    O, LSE = oracle.forward(p)
    sig = 1.0 / (1.0 + math.exp(s - t))
    np.testing.assert_allclose(O[0, 0, 0], sig * v[0, 0, 0], rtol=1e-15)
    assert LSE[0, 0, 0] == pytest.approx(math.log(math.exp(t) + math.exp(s)), rel=1e-15)
    g = oracle.backward(p, dO, O, LSE)
    p0 = 1 - sig
    assert g["dsink"][0] == pytest.approx(-p0 * float(dO[0, 0, 0] @ O[0, 0, 0]), rel=1e-14)
    np.testing.assert_allclose(g["dv"][0, 0, 0], sig * dO[0, 0, 0], rtol=1e-14)


def test_sink_limits():
    """sink -> -inf is no sink (bit-identical); a very large sink drives O to 0."""
    p, dO = full_problem(S=7, sink=False)
    O0, L0 = oracle.forward(p)
    p.sink = np.full((p.Hq,), -1e4)
    O1, L1 = oracle.forward(p)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    p.sink = np.full((p.Hq,), 1e3)
    O2, L2 = oracle.forward(p)
    assert np.max(np.abs(O2)) < 1e-300 and np.allclose(L2, 1e3)


def test_off_by_one_equals_sdpa_with_a_zero_key():
    """The off-by-one softmax -- one extra column of logit 0 in every row, the "off-by-one"
    softmax type TransformerEngine PR #3551 tests beside "learnable" -- is the oracle's sink
    held at 0.  It equals plain attention over the keys plus one all-zero key (logit 0 under
    any scale) with an all-zero value that every query sees: torch SDPA in fp64, with
    autograd for dq, dk, dv."""
    F = torch.nn.functional
    r = rng(11)
    B, S, H, D, scale = 2, 9, 2, 4, 0.5
    q, k, v = r.normal(0, 1.5, (B, S, H, D)), r.normal(0, 1.5, (B, S, H, D)), r.normal(0, 1, (B, S, H, D))
    dO = r.normal(0, 1, (B, S, H, D))
    for causal in (False, True):
        p = Problem(q, k, v, scale=scale, causal=causal, sink=np.zeros(H))
        O, LSE = oracle.forward(p)
        g = oracle.backward(p, dO, O, LSE)
        qt, kt, vt = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v))
        zero = torch.zeros(B, H, 1, D, dtype=torch.float64)
        mask = torch.ones(S, S + 1, dtype=torch.bool)
        if causal:
            mask[:, :S] = torch.tril(torch.ones(S, S, dtype=torch.bool))
        out = F.scaled_dot_product_attention(qt, torch.cat([kt, zero], 2), torch.cat([vt, zero], 2),
                                             attn_mask=mask, scale=scale)
        (out * torch.tensor(dO).permute(0, 2, 1, 3)).sum().backward()
        t = lambda x: x.detach().permute(0, 2, 1, 3).numpy()
        assert rel(O, t(out)) < 1e-13
        assert rel(g["dq"], t(qt.grad)) < 1e-12
        assert rel(g["dk"], t(kt.grad)) < 1e-12
        assert rel(g["dv"], t(vt.grad)) < 1e-12


def test_dsink_two_ways():
    """dsink equals -sum p0 D with p0 = exp(sink - LSE) and D = dO.O computed here, and
    the sum runs over every batch and row."""
    p, dO = full_problem(S=7, B=2)
    O, LSE = oracle.forward(p)
    g = oracle.backward(p, dO, O, LSE)
    D = np.einsum("bihd,bihd->bhi", dO, O)
    expect = -(np.exp(p.sink[None, :, None] - LSE) * D).sum(axis=(0, 2))
    np.testing.assert_allclose(g["dsink"], expect, rtol=1e-13)


def test_sink_once_tile_merge_matches_unsplit():
    """Split the keys in two tiles, run the oracle on each, give only the first tile the sink,
    merge (O, LSE) by log-sum-exp: the result equals the unsplit oracle (the sink entering
    each row exactly once).  Giving both tiles the sink does not."""
    tol = FIG["sink_once_schedule_match"]["abs_tol"]
    r = rng(5)
    B, S, Hq, D = 1, 16, 2, 4
    q, k, v = r.normal(0, 1, (B, S, Hq, D)), r.normal(0, 1, (B, S, Hq, D)), r.normal(0, 1, (B, S, Hq, D))
    sink = r.normal(0, 5, (Hq,))
    full = Problem(q, k, v, scale=0.5, softcap=3.0, sink=sink)
    O, LSE = oracle.forward(full)
    h = S // 2
    t0 = Problem(q, k[:, :h], v[:, :h], scale=0.5, softcap=3.0, sink=sink)
    t1 = Problem(q, k[:, h:], v[:, h:], scale=0.5, softcap=3.0)
    t1s = Problem(q, k[:, h:], v[:, h:], scale=0.5, softcap=3.0, sink=sink)
    O0, L0 = oracle.forward(t0)
    for tile1, ok in ((t1, True), (t1s, False)):
        O1, L1 = oracle.forward(tile1)
        L = np.logaddexp(L0, L1)
        w0 = np.exp(L0 - L).transpose(0, 2, 1)[..., None]
        w1 = np.exp(L1 - L).transpose(0, 2, 1)[..., None]
        Om = w0 * O0 + w1 * O1
        err = max(np.max(np.abs(Om - O)), np.max(np.abs(L - LSE)))
        assert (err <= 20 * tol) == ok, err


# ----------------------------------------------------------------- GQA, masks

def test_gqa_equals_mha_on_repeated_kv():
    """GQA with G = Hq/Hkv equals MHA on K, V repeated per group; dK/dV are the group sums."""
    r = rng(6)
    B, S, Hq, Hkv, D = 2, 9, 6, 2, 4
    q = r.normal(0, 1, (B, S, Hq, D))
    k, v = r.normal(0, 1, (B, S, Hkv, D)), r.normal(0, 1, (B, S, Hkv, D))
    dO = r.normal(0, 1, (B, S, Hq, D))
    sink = r.normal(0, 2, (Hq,))
    kw = dict(scale=0.5, causal=True, softcap=2.0, sink=sink)
    pg = Problem(q, k, v, **kw)
    pm = Problem(q, np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2), **kw)
    Og, Lg = oracle.forward(pg)
    Om, Lm = oracle.forward(pm)
    assert np.array_equal(Og, Om) and np.array_equal(Lg, Lm)
    gg = oracle.backward(pg, dO, Og, Lg)
    gm = oracle.backward(pm, dO, Om, Lm)
    G = Hq // Hkv
    for key in ("dk", "dv"):
        summed = gm[key].reshape(B, S, Hkv, G, D).sum(axis=3)
        np.testing.assert_allclose(gg[key], summed, rtol=1e-13, atol=1e-15)
    assert np.array_equal(gg["dq"], gm["dq"])
    np.testing.assert_allclose(gg["dsink"], gm["dsink"], rtol=1e-14)


def test_window_covering_sequence_equals_causal():
    p, dO = full_problem(S=7, window=0)
    O0, L0 = oracle.forward(p)
    p.window = 7
    O1, L1 = oracle.forward(p)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_single_segment_equals_none():
    p, dO = full_problem(S=7, segs=False)
    O0, L0 = oracle.forward(p)
    g0 = oracle.backward(p, dO, O0, L0)
    p.seg_q = p.seg_k = np.zeros((1, 7), np.int32)
    O1, L1 = oracle.forward(p)
    g1 = oracle.backward(p, dO, O1, L1)
    assert np.array_equal(O0, O1)
    for key in ("dq", "dk", "dv", "dbias", "dsink"):
        assert np.array_equal(g0[key], g1[key]), key


def test_cross_segment_perturbation_leaves_other_segment_bit_identical():
    """Changing q, k, v, dO of segment 1 leaves segment 0's outputs and gradients unchanged."""
    p, dO = full_problem(S=7, sink=False, bias=False)
    seg0 = p.seg_q[0] == 0
    O0, L0 = oracle.forward(p)
    g0 = oracle.backward(p, dO, O0, L0)
    r = rng(9)
    for arr in (p.q, p.k, p.v, dO):
        arr[:, ~seg0] = r.normal(0, 3, arr[:, ~seg0].shape)
    O1, L1 = oracle.forward(p)
    g1 = oracle.backward(p, dO, O1, L1)
    assert np.array_equal(O0[:, seg0], O1[:, seg0]) and np.array_equal(L0[..., seg0], L1[..., seg0])
    for key in ("dq", "dk", "dv"):
        assert np.array_equal(g0[key][:, seg0], g1[key][:, seg0]), key


def _count(S, Sk=None, causal=False, window=0, seg=None, B=1, Hq=1):
    Sk = S if Sk is None else Sk
    z = np.zeros
    p = Problem(z((B, S, Hq, 1)), z((B, Sk, 1, 1)), z((B, Sk, 1, 1)), scale=1.0,
                causal=causal, window=window, seg_q=seg, seg_k=seg)
    return oracle.count_visible(p)


def test_visible_pair_counts_closed_forms():
    S = 37
    assert _count(S) == S * S
    assert _count(S, causal=True) == S * (S + 1) // 2
    W = 10
    assert _count(S, causal=True, window=W) == sum(min(i + 1, W) for i in range(S))
    assert _count(S, window=W) == sum(S - max(0, i - W + 1) for i in range(S))
    lens = [5, 13, 19]
    seg = np.repeat(np.arange(3, dtype=np.int32), lens)[None]
    assert _count(S, causal=True, seg=seg) == sum(L * (L + 1) // 2 for L in lens)
    assert _count(S, seg=seg) == sum(L * L for L in lens)
    # bottom-right causal with Sq < Sk: query i sees keys 0 .. i + Sk - Sq
    assert _count(5, Sk=9, causal=True) == sum(i + 4 + 1 for i in range(5))
    # Windows with Sq != Sk, counted by hand from the bottom-right reading (query i stands at
    # key position i + Sk - Sq and sees the W keys ending there; without causal, every key
    # from that window's start to the end).  Sq = 5, Sk = 9, W = 3: every row sees 3 keys
    # causally; without causal row i sees keys i + 2 .. 8, i.e. 7, 6, 5, 4, 3.
    assert _count(5, Sk=9, causal=True, window=3) == 15
    assert _count(5, Sk=9, window=3) == 25
    # Sq = 9, Sk = 5, W = 2: query i stands at i - 4.  Causal: rows 0-3 see nothing, row 4
    # sees key 0, rows 5-8 see two keys each.  Without causal: row i sees keys i - 5 .. 4,
    # i.e. 5 for rows 0-5 and then 4, 3, 2.
    assert _count(9, Sk=5, causal=True, window=2) == 9
    assert _count(9, Sk=5, window=2) == 5 * 6 + 4 + 3 + 2
    assert _count(S, causal=True, B=2, Hq=3) == 6 * S * (S + 1) // 2


def test_visible_pairs_with_ids_per_axis():
    """Ids given per axis with Sq != Sk (a chunk of queries at the end of a packed key row):
    query i stands at key position i + Sk - Sq and sees the keys of its own id up to there.
    Sq = 4, Sk = 7, query ids [1, 1, 2, 2], key ids [0, 0, 1, 1, 1, 2, 2], counted by hand:
    causal rows see keys {2, 3}, {2, 3, 4}, {5}, {5, 6} (8 pairs); without causal every id-1
    row sees 3 keys and every id-2 row 2 (10 pairs).  Reading a query's id from the key array
    (or the other way round) gives 10 causal pairs instead."""
    z = np.zeros
    seg_q = np.array([[1, 1, 2, 2]], np.int32)
    seg_k = np.array([[0, 0, 1, 1, 1, 2, 2]], np.int32)
    for causal, want in ((True, 8), (False, 10)):
        p = Problem(z((1, 4, 1, 1)), z((1, 7, 1, 1)), z((1, 7, 1, 1)), scale=1.0, causal=causal,
                    seg_q=seg_q, seg_k=seg_k)
        assert oracle.count_visible(p) == want, causal
    p = Problem(z((1, 4, 1, 1)), z((1, 7, 1, 1)), z((1, 7, 1, 1)), scale=1.0, causal=True, seg_q=seg_q, seg_k=seg_k)
    count, first, last = oracle.row_visible(p)
    assert count.tolist() == [[2, 3, 1, 2]] and first.tolist() == [[2, 2, 5, 5]] and last.tolist() == [[3, 4, 5, 6]]
    count, first, last = oracle.col_visible(p)
    assert count.tolist() == [[0, 0, 2, 2, 1, 2, 1]]
    assert first.tolist() == [[-1, -1, 0, 0, 1, 2, 3]] and last.tolist() == [[-1, -1, 1, 1, 1, 3, 3]]


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 3), (False, 3)])
def test_bottom_right_alignment_equals_square_problem(causal, window):
    """With Sq < Sk, query i of the short problem is query i + Sk - Sq of the square problem on
    the same keys (extra queries in front); with Sq > Sk under causal masking, queries past
    Sq - Sk are the square problem's on their own keys and the leading ones see nothing.  The
    square case is pinned above (closed-form counts, finite differences), so these fix the
    alignment of the causal and window terms when the lengths differ: O, LSE and every
    gradient."""
    r = rng(21)
    D, Hq, Hkv, Sq, Sk = 4, 2, 1, 5, 9
    off = Sk - Sq
    k = r.normal(0, 1.5, (1, Sk, Hkv, D))
    v = r.normal(0, 1, (1, Sk, Hkv, D))
    q_sq = r.normal(0, 1.5, (1, Sk, Hq, D))
    dO_sq = r.normal(0, 1, (1, Sk, Hq, D))
    kw = dict(scale=0.5, causal=causal, window=window, softcap=3.0, sink=r.normal(0, 1, (Hq,)))
    square = Problem(q_sq, k, v, **kw)
    short = Problem(q_sq[:, off:].copy(), k, v, **kw)
    Os, Ls = oracle.forward(square)
    O, L = oracle.forward(short)
    np.testing.assert_allclose(O, Os[:, off:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(L, Ls[:, :, off:], rtol=0, atol=1e-13)
    # gradients: dO zero on the square problem's extra queries, so only the shared ones count
    dO_sq[:, :off] = 0.0
    gs = oracle.backward(square, dO_sq, Os, Ls)
    g = oracle.backward(short, dO_sq[:, off:].copy(), O, L)
    np.testing.assert_allclose(g["dq"], gs["dq"][:, off:], rtol=0, atol=1e-13)
    for key in ("dk", "dv", "dsink"):
        np.testing.assert_allclose(g[key], gs[key], rtol=0, atol=1e-13)
    if not causal:
        return
    # Sq > Sk: the keys are the square problem's first Sq - off ... swap the roles: 9 queries
    # against 5 keys; rows 4.. equal the 5 x 5 problem on those rows, rows 0..3 see nothing.
    k5, v5 = k[:, :Sq], v[:, :Sq]
    q9 = r.normal(0, 1.5, (1, Sk, Hq, D))
    tall = Problem(q9, k5, v5, **kw)
    sq5 = Problem(q9[:, off:].copy(), k5, v5, **kw)
    Ot, Lt = oracle.forward(tall)
    O5, L5 = oracle.forward(sq5)
    np.testing.assert_allclose(Ot[:, off:], O5, rtol=0, atol=1e-14)
    np.testing.assert_allclose(Lt[:, :, off:], L5, rtol=0, atol=1e-13)
    assert np.all(Ot[:, :off] == 0)
    np.testing.assert_allclose(Lt[:, :, :off], np.broadcast_to(kw["sink"][:, None], (Hq, off))[None],
                               rtol=0, atol=1e-15)


def test_row_and_column_extents_brute_force():
    """Per-row and per-key visible counts and extents: equal to enumerating oracle.visible pair
    by pair on tiny shapes (causal + window + sorted and unsorted segments, Sq != Sk), and the
    counts sum to count_visible (pinned by the closed forms above)."""
    for Sq, Sk, causal, window, seg_kind in [(9, 9, True, 4, "runs"), (7, 11, True, 3, None),
                                             (11, 6, False, 2, None), (10, 10, True, 0, "interleaved")]:
        z = np.zeros
        kw = dict(scale=1.0, causal=causal, window=window)
        if seg_kind == "runs":
            kw["seg_q"] = kw["seg_k"] = np.array([[0, 0, 0, 1, 1, 2, 2, 2, 2]], np.int32)
        elif seg_kind == "interleaved":
            kw["seg_q"] = kw["seg_k"] = (np.arange(Sq, dtype=np.int32) % 3)[None]
        p = Problem(z((1, Sq, 1, 1)), z((1, Sk, 1, 1)), z((1, Sk, 1, 1)), **kw)
        vis = np.array([[oracle.visible(p, 0, i, j) for j in range(Sk)] for i in range(Sq)])
        rc, rf, rl = oracle.row_visible(p)
        cc, cf, cl = oracle.col_visible(p)
        for i in range(Sq):
            js = np.flatnonzero(vis[i])
            assert rc[0, i] == len(js)
            assert (rf[0, i], rl[0, i]) == ((js[0], js[-1]) if len(js) else (-1, -1))
        for j in range(Sk):
            is_ = np.flatnonzero(vis[:, j])
            assert cc[0, j] == len(is_)
            assert (cf[0, j], cl[0, j]) == ((is_[0], is_[-1]) if len(is_) else (-1, -1))
        assert rc.sum() == cc.sum() == oracle.count_visible(p)


def test_bias_gradient_follows_bias_broadcast_shape():
    """dbias has the bias's own shape: broadcast over batch it is the sum of the per-batch
    gradients; broadcast over heads, the sum over heads."""
    r = rng(10)
    B, S, H, D = 2, 6, 3, 4
    q, k, v, dO = (r.normal(0, 1, (B, S, H, D)) for _ in range(4))
    kw = dict(scale=0.5, causal=True, softcap=3.0)
    full = r.normal(0, 1, (B, H, S, S))
    pf = Problem(q, k, v, bias=full, **kw)
    Of, Lf = oracle.forward(pf)
    gf = oracle.backward(pf, dO, Of, Lf)
    shared_b = np.broadcast_to(full[:1], full.shape).copy()
    pb = Problem(q, k, v, bias=full[:1], **kw)
    pbe = Problem(q, k, v, bias=shared_b, **kw)
    Ob, Lb = oracle.forward(pb)
    gb = oracle.backward(pb, dO, Ob, Lb)
    Obe, Lbe = oracle.forward(pbe)
    gbe = oracle.backward(pbe, dO, Obe, Lbe)
    assert gb["dbias"].shape == (1, H, S, S)
    np.testing.assert_allclose(gb["dbias"][0], gbe["dbias"].sum(0), rtol=1e-13, atol=1e-16)
    ph = Problem(q, k, v, bias=full[:, :1], **kw)
    phe = Problem(q, k, v, bias=np.broadcast_to(full[:, :1], full.shape).copy(), **kw)
    gh = oracle.backward(ph, dO, *oracle.forward(ph))
    ghe = oracle.backward(phe, dO, *oracle.forward(phe))
    assert gh["dbias"].shape == (B, 1, S, S)
    np.testing.assert_allclose(gh["dbias"][:, 0], ghe["dbias"].sum(1), rtol=1e-13, atol=1e-16)
    assert gf["dbias"].shape == (B, H, S, S)


def test_fully_masked_row_without_and_with_sink():
    """A query whose segment has no key: no sink -> O = 0, LSE = -inf, zero dQ;
    with a sink -> LSE = sink, O = 0."""
    S = 4
    r = rng(11)
    q, k, v = (r.normal(0, 1, (1, S, 1, 2)) for _ in range(3))
    seg_q = np.array([[0, 0, 1, 1]], np.int32)
    seg_k = np.array([[0, 0, 0, 0]], np.int32)
    dO = r.normal(0, 1, (1, S, 1, 2))
    p = Problem(q, k, v, scale=1.0, seg_q=seg_q, seg_k=seg_k)
    O, L = oracle.forward(p)
    assert np.all(O[0, 2:] == 0) and np.all(np.isneginf(L[0, 0, 2:]))
    g = oracle.backward(p, dO, O, L)
    assert np.all(g["dq"][0, 2:] == 0)
    p.sink = np.array([0.7])
    O, L = oracle.forward(p)
    assert np.all(O[0, 2:] == 0) and np.allclose(L[0, 0, 2:], 0.7)


# ----------------------------------------------------------------- tile schedule

def _blockwise_forward(p, BM, BN):
    """Online softmax over KV tiles of BN keys for row blocks of BM rows, with the sink folded
    into the initial running state (m = sink, l = 1) -- the schedule the GPU kernels use."""
    B, Sq, Sk, Hq, D = p.B, p.Sq, p.Sk, p.Hq, p.D
    G = p.Hq // p.Hkv
    O = np.zeros((B, Sq, Hq, D))
    LSE = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i0 in range(0, Sq, BM):
                rows = np.arange(i0, min(i0 + BM, Sq))
                m = np.full(len(rows), -np.inf if p.sink is None else p.sink[h])
                l = np.zeros(len(rows)) if p.sink is None else np.ones(len(rows))
                acc = np.zeros((len(rows), D))
                for j0 in range(0, Sk, BN):
                    cols = np.arange(j0, min(j0 + BN, Sk))
                    u = p.scale * p.q[b, rows, h] @ p.k[b, cols, g].T
                    t = p.softcap * np.tanh(u / p.softcap) if p.softcap else u
                    vis = np.array([[oracle.visible(p, b, i, j) for j in cols] for i in rows])
                    t = np.where(vis, t, -np.inf)
                    mn = np.maximum(m, t.max(axis=1))
                    alpha = np.where(np.isneginf(mn), 0.0, np.exp(m - mn))
                    pt = np.where(vis, np.exp(t - mn[:, None]), 0.0)
                    l = alpha * l + pt.sum(axis=1)
                    acc = alpha[:, None] * acc + pt @ p.v[b, cols, g]
                    m = mn
                O[b, rows, h] = acc / np.where(l > 0, l, 1.0)[:, None]
                LSE[b, h, rows] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, LSE


@pytest.mark.parametrize("BM,BN", [(64, 64), (64, 128), (128, 64)])
def test_tile_schedule_emulation_matches_oracle(BM, BN):
    r = rng(12)
    B, S, Hq, Hkv, D = 1, 150, 2, 1, 4
    q, k, v = r.normal(0, 2, (B, S, Hq, D)), r.normal(0, 2, (B, S, Hkv, D)), r.normal(0, 1, (B, S, Hkv, D))
    seg = np.repeat(np.arange(3, dtype=np.int32), [70, 33, 47])[None]
    p = Problem(q, k, v, scale=0.5, causal=True, window=90, softcap=3.0,
                sink=r.normal(0, 5, (Hq,)), seg_q=seg)
    O, LSE = oracle.forward(p)
    Oe, Le = _blockwise_forward(p, BM, BN)
    assert np.max(np.abs(Oe - O)) <= 1e-13 and np.max(np.abs(Le - LSE)) <= 1e-13


def test_row_and_column_selection_equals_full_backward():
    """Selecting rows / columns in the backward returns exactly the full backward's values on
    them (and the selection masks stay alive while the C code reads them)."""
    p, dO = full_problem(S=7, B=2)
    O, LSE = oracle.forward(p)
    full = oracle.backward(p, dO, O, LSE)
    for _ in range(20):
        part = oracle.backward(p, dO, O, LSE, rows=[1, 4, 6], cols=[0, 5])
        assert np.array_equal(part["dq"][:, [1, 4, 6]], full["dq"][:, [1, 4, 6]])
        assert np.array_equal(part["dk"][:, [0, 5]], full["dk"][:, [0, 5]])
        assert np.array_equal(part["dv"][:, [0, 5]], full["dv"][:, [0, 5]])
        assert np.all(np.isnan(part["dq"][:, [0, 2, 3, 5]]))
