"""The kernels' soft-cap reciprocal r = 1 / (1 + 2^x), emulated in float32 on the host: the
bit-level seed (a constant minus the bits of d) and two Newton-Raphson steps, as compiled into
tc_common.cuh.  Checks the error bound the kernels' comments state, the one-sided error, and
that the clamp keeps every x finite."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "attention_flash_attn_gb300", "csrc", "tc_common.cuh")


def _source_constant():
    body = open(SRC).read().split("f2_sigmoid2_neg(uint64_t x2, uint64_t &e2)", 1)[1].split("\n}\n", 1)[0]
    (k,) = re.findall(r"0x([0-9A-Fa-f]{8})u - __float_as_uint\(na\)", body)
    steps = body.count("r = f2_fma(r, f2_fma(nd, r, one), r);")
    (clamp,) = re.findall(r"fminf\(xa, ([0-9.]+)f\)", body)
    return int(k, 16), steps, float(clamp)


def emulate(x):
    """float32 emulation with exact 2^x (the kernels use ex2.approx, error ~2 ulp)."""
    k, steps, clamp = _source_constant()
    x = np.minimum(np.asarray(x, dtype=np.float32), np.float32(clamp))
    e = np.exp2(x.astype(np.float64)).astype(np.float32)
    nd = (e * np.float32(-1) + np.float32(-1)).astype(np.float32)
    r = ((np.uint32(k) - nd.view(np.uint32)) & np.uint32(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    one = np.float32(1)
    for _ in range(steps):
        r = (r * (nd * r + one) + r).astype(np.float32)
    return r


def test_source_form():
    k, steps, clamp = _source_constant()
    assert k == 0xFEF311C0 and steps == 2 and clamp == 126.0


def test_relative_error_and_sign():
    x = np.concatenate([np.linspace(-160, 200, 400001), np.linspace(-2, 2, 100001)]).astype(np.float32)
    r = emulate(x).astype(np.float64)
    xc = np.minimum(x.astype(np.float64), 126.0)
    exact = 1.0 / (1.0 + np.exp2(xc))
    assert np.all(np.isfinite(r))
    big = exact > 1e-30  # below that, flushed seeds give 0 (tanh = 1 exactly in fp32)
    rel = np.abs(r[big] - exact[big]) / exact[big]
    assert rel.max() < 7e-6, rel.max()
    # Newton's iteration for a reciprocal approaches from below (plus fp32 rounding)
    assert np.all(r[big] <= exact[big] * (1 + 2e-7))
    assert np.all(r[~big] <= 1e-30)


def test_capped_logit_error_bound():
    """t = cap (1 - 2 r): |error| <= 2 cap r 7e-6, so at most 7e-4 for cap 50."""
    cap = 50.0
    u = np.linspace(-400, 400, 200001)
    x = (2 * u / cap * np.log2(np.e)).astype(np.float32)
    t = cap * (1 - 2 * emulate(x).astype(np.float64))
    err = np.abs(t - cap * np.tanh(u / cap))
    assert err.max() < 7.5e-4, err.max()
