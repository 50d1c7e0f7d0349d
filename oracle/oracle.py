"""ctypes marshalling for the fp64 oracle in ``attn_oracle.c`` (test infrastructure only).

No arithmetic of the method happens here: every quantity is computed by the C
functions, which follow the definition in that file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc (fp64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _CProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Sq", ctypes.c_int), ("Sk", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("bias", ctypes.c_void_p), ("bias_B", ctypes.c_int), ("bias_H", ctypes.c_int),
        ("seg_q", ctypes.c_void_p), ("seg_k", ctypes.c_void_p),
        ("causal", ctypes.c_int), ("window", ctypes.c_int),
        ("softcap", ctypes.c_double), ("sink", ctypes.c_void_p), ("scale", ctypes.c_double),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_CProblem)
        vp = ctypes.c_void_p
        lib.oracle_forward.argtypes = [P, vp, vp, vp]
        lib.oracle_rowdot.argtypes = [P, vp, vp, vp]
        lib.oracle_backward_dq.argtypes = [P, vp, vp, vp, vp, vp]
        lib.oracle_backward_dkdv.argtypes = [P, vp, vp, vp, vp, vp, vp]
        lib.oracle_backward_dbias.argtypes = [P, vp, vp, vp, vp]
        lib.oracle_backward_dsink.argtypes = [P, vp, vp, vp]
        lib.oracle_count_visible.argtypes = [P, ctypes.c_int]
        lib.oracle_count_visible.restype = ctypes.c_longlong
        lib.oracle_visible.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        ll, ip = ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_int)
        lib.oracle_row_visible.argtypes = [P, ctypes.c_int, ctypes.c_int, ll, ip, ip]
        lib.oracle_col_visible.argtypes = [P, ctypes.c_int, ctypes.c_int, ll, ip, ip]
        lib.oracle_capped.argtypes = [P, ctypes.c_double]
        lib.oracle_capped.restype = ctypes.c_double
        lib.oracle_cap_factor.argtypes = [P, ctypes.c_double]
        lib.oracle_cap_factor.restype = ctypes.c_double
        _lib = lib
    return _lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


@dataclass
class Problem:
    """One attention problem in fp64.

    q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D]; bias [Bb,Hb,Sq,Sk] (Bb in {1,B}, Hb in {1,Hq}) or None;
    seg_q [B,Sq] / seg_k [B,Sk] int32 or None; sink [Hq] or None; softcap 0 = off.
    """
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    scale: float
    causal: bool = False
    window: int = 0
    softcap: float = 0.0
    bias: Optional[np.ndarray] = None
    sink: Optional[np.ndarray] = None
    seg_q: Optional[np.ndarray] = None
    seg_k: Optional[np.ndarray] = None

    def __post_init__(self):
        self.q, self.k, self.v = _f64(self.q), _f64(self.k), _f64(self.v)
        self.bias, self.sink = _f64(self.bias), _f64(self.sink)
        if self.seg_q is not None:
            self.seg_q = np.ascontiguousarray(self.seg_q, dtype=np.int32)
            self.seg_k = np.ascontiguousarray(
                self.seg_q if self.seg_k is None else self.seg_k, dtype=np.int32)
        B, Sq, Hq, D = self.q.shape
        _, Sk, Hkv, _ = self.k.shape
        assert self.k.shape == (B, Sk, Hkv, D) and self.v.shape == (B, Sk, Hkv, D)
        assert Hq % Hkv == 0
        self.B, self.Sq, self.Sk, self.Hq, self.Hkv, self.D = B, Sq, Sk, Hq, Hkv, D
        if self.bias is not None:
            assert self.bias.ndim == 4 and self.bias.shape[2:] == (Sq, Sk)
            assert self.bias.shape[0] in (1, B) and self.bias.shape[1] in (1, Hq)

    def _c(self) -> _CProblem:
        c = _CProblem()
        c.B, c.Sq, c.Sk, c.Hq, c.Hkv, c.D = self.B, self.Sq, self.Sk, self.Hq, self.Hkv, self.D
        c.q, c.k, c.v = _ptr(self.q), _ptr(self.k), _ptr(self.v)
        c.bias = _ptr(self.bias)
        c.bias_B = 1 if self.bias is None or self.bias.shape[0] == 1 else self.B
        c.bias_H = 1 if self.bias is None or self.bias.shape[1] == 1 else self.Hq
        c.seg_q, c.seg_k = _ptr(self.seg_q), _ptr(self.seg_k)
        c.causal, c.window = int(bool(self.causal)), int(self.window)
        c.softcap, c.sink, c.scale = float(self.softcap), _ptr(self.sink), float(self.scale)
        return c


def _mask(m, n):
    if m is None:
        return None
    a = np.zeros(n, dtype=np.uint8)
    a[np.asarray(m)] = 1
    return a


def forward(p: Problem, rows=None):
    """O [B,Sq,Hq,D] and LSE [B,Hq,Sq] (fp64).  ``rows``: query indices to compute
    (all when None); entries of other rows are NaN."""
    lib = _load()
    O = np.full((p.B, p.Sq, p.Hq, p.D), np.nan)
    LSE = np.full((p.B, p.Hq, p.Sq), np.nan)
    rm = _mask(rows, p.Sq)
    c = p._c()
    lib.oracle_forward(ctypes.byref(c), _ptr(rm), _ptr(O), _ptr(LSE))
    return O, LSE


def rowdot(p: Problem, dO, O):
    """D_i = dO_i . O_i  [B,Hq,Sq]."""
    lib = _load()
    dO, O = _f64(dO), _f64(O)
    Dv = np.empty((p.B, p.Hq, p.Sq))
    c = p._c()
    lib.oracle_rowdot(ctypes.byref(c), _ptr(dO), _ptr(O), _ptr(Dv))
    return Dv


def backward(p: Problem, dO, O, LSE, rows=None, cols=None, want=("dq", "dk", "dv", "dbias", "dsink")):
    """Analytic backward in fp64.

    O and LSE come from ``forward`` on the same problem.  ``rows`` restricts dQ to those
    query rows (LSE/O need only be valid there); dK/dV/dbias/dsink need every row of O and
    LSE.  ``cols`` restricts dK/dV to those key columns.  Returns a dict with the requested
    gradients (unrequested or inapplicable ones are None); unselected entries are NaN.
    """
    lib = _load()
    dO, O, LSE = _f64(dO), _f64(O), _f64(LSE)
    c = p._c()
    Dv = np.nan_to_num(rowdot(p, dO, np.nan_to_num(O)), nan=0.0)
    out = {"D": Dv}
    # masks are bound to names so they outlive the C calls that read them
    row_mask, col_mask = _mask(rows, p.Sq), _mask(cols, p.Sk)
    if "dq" in want:
        dQ = np.full(p.q.shape, np.nan)
        lib.oracle_backward_dq(ctypes.byref(c), _ptr(dO), _ptr(LSE), _ptr(Dv),
                               _ptr(row_mask), _ptr(dQ))
        out["dq"] = dQ
    if "dk" in want or "dv" in want:
        dK = np.full(p.k.shape, np.nan)
        dV = np.full(p.v.shape, np.nan)
        lib.oracle_backward_dkdv(ctypes.byref(c), _ptr(dO), _ptr(LSE), _ptr(Dv),
                                 _ptr(col_mask), _ptr(dK), _ptr(dV))
        out["dk"], out["dv"] = dK, dV
    out["dbias"] = None
    if "dbias" in want and p.bias is not None:
        db = np.full(p.bias.shape, np.nan)
        lib.oracle_backward_dbias(ctypes.byref(c), _ptr(dO), _ptr(LSE), _ptr(Dv), _ptr(db))
        out["dbias"] = db
    out["dsink"] = None
    if "dsink" in want and p.sink is not None:
        ds = np.empty(p.Hq)
        lib.oracle_backward_dsink(ctypes.byref(c), _ptr(LSE), _ptr(Dv), _ptr(ds))
        out["dsink"] = ds
    return out


def count_visible(p: Problem) -> int:
    """Brute-force count of visible (b, h, i, j) pairs (the mask definition, pair by pair)."""
    lib = _load()
    c = p._c()
    return int(sum(lib.oracle_count_visible(ctypes.byref(c), b) for b in range(p.B)) * p.Hq)


def visible(p: Problem, b: int, i: int, j: int) -> bool:
    lib = _load()
    c = p._c()
    return bool(lib.oracle_visible(ctypes.byref(c), b, i, j))


def capped(p: Problem, u: float) -> float:
    lib = _load()
    c = p._c()
    return lib.oracle_capped(ctypes.byref(c), float(u))


def cap_factor(p: Problem, u: float) -> float:
    lib = _load()
    c = p._c()
    return lib.oracle_cap_factor(ctypes.byref(c), float(u))


def _extents(p: Problem, fn, n):
    lib = _load()
    c = p._c()
    count = np.zeros((p.B, n), np.int64)
    first = np.zeros((p.B, n), np.int64)
    last = np.zeros((p.B, n), np.int64)
    cn, cf, cl = ctypes.c_longlong(), ctypes.c_int(), ctypes.c_int()
    f = getattr(lib, fn)
    for b in range(p.B):
        for x in range(n):
            f(ctypes.byref(c), b, x, ctypes.byref(cn), ctypes.byref(cf), ctypes.byref(cl))
            count[b, x], first[b, x], last[b, x] = cn.value, cf.value, cl.value
    return count, first, last


def row_visible(p: Problem):
    """Per query row: (number of visible keys, first, last) as [B, Sq] arrays (-1: none)."""
    return _extents(p, "oracle_row_visible", p.Sq)


def col_visible(p: Problem):
    """Per key: (number of queries that see it, first, last) as [B, Sk] arrays (-1: none)."""
    return _extents(p, "oracle_col_visible", p.Sk)
