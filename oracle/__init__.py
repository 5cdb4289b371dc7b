"""CPU oracle for exhaustive SIFT descriptor matching -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and it shares no code with it.

The arithmetic lives in ``serac_oracle.c`` (plain brute force, OpenMP over rows or
columns).  This module only builds that file with gcc and marshals numpy arrays.
What it computes, with the passages it follows, is stated at the top of the C file.

Parity status: every exported function is pinned by ``tests/test_oracle_pins.py``
(hand-worked examples, an independent numpy brute force on tiny inputs, planted
correspondence recovery, symmetry, ratio-test and gate boundaries).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "serac_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

GCC_FLAGS = ["-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11"]


def build_library(force: bool = False) -> str:
    """Compile serac_oracle.c into liboracle.so (in place) when missing or stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, _SRC, "-o", tmp], check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [("ratio_num_sq", ctypes.c_int64), ("ratio_den_sq", ctypes.c_int64),
                ("norm_sq", ctypes.c_int64), ("min_score", ctypes.c_int64),
                ("mutual", ctypes.c_int32), ("col_ratio", ctypes.c_int32),
                ("max_features", ctypes.c_int32)]


@dataclass(frozen=True)
class Params:
    """Matching parameters in exact integers (see the C file for their meaning)."""
    ratio_num_sq: int = 16
    ratio_den_sq: int = 25
    norm_sq: int = 512 * 512
    min_score: int = 200499
    mutual: int = 1
    col_ratio: int = 1
    max_features: int = 0  # K > 0: each image takes part with its first K descriptors

    def _c(self) -> _Params:
        return _Params(self.ratio_num_sq, self.ratio_den_sq, self.norm_sq,
                       self.min_score, self.mutual, self.col_ratio, self.max_features)


def default_params(max_ratio: float = 0.8, max_angle: float = 0.7,
                   mutual: int = 1, col_ratio: int = 1, max_features: int = 0) -> Params:
    """0.8 / 0.7 rad -> r^2 = 16/25 and min_score = ceil(cos(0.7) * 512^2) = 200499.

    max_ratio is read to 4 decimals (r = R / 10^4) and r^2 = R^2 / 10^8 is reduced.
    """
    n = 512 * 512
    r = int(round(max_ratio * 10000))
    num, den = r * r, 10 ** 8
    g = math.gcd(num, den) if num else den
    return Params(num // g, den // g, n, int(math.ceil(math.cos(max_angle) * n)),
                  mutual, col_ratio, max_features)


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_library())
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.oracle_scores.argtypes = [P, i32, P, i32, P]
        lib.oracle_row_top2.argtypes = [P, i32, P, i32, P, i32, P]
        lib.oracle_col_top2.argtypes = [P, i32, P, i32, P, i32, P]
        lib.oracle_match.argtypes = [P, i32, P, i32, ctypes.POINTER(_Params), P, P, P, i32, P]
        lib.oracle_accept_rows.argtypes = [P, i32, P, i32, ctypes.POINTER(_Params), P, i32, P, P, P]
        lib.oracle_row_topk.argtypes = [P, i32, P, i32, i32, P, i32, P, P]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _u8(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint8)
    if x.ndim != 2 or x.shape[1] != 128:
        raise ValueError("descriptors must be (n, 128) uint8")
    return x


def _ptr(x):
    return None if x is None else x.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def scores(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Full integer score matrix (nA, nB), small inputs only."""
    a, b = _u8(a), _u8(b)
    out = np.zeros((a.shape[0], b.shape[0]), np.int32)
    rc = _load().oracle_scores(_ptr(a), a.shape[0], _ptr(b), b.shape[0], _ptr(out))
    assert rc == 0
    return out


def row_top2(a: np.ndarray, b: np.ndarray, rows=None) -> np.ndarray:
    """(n, 4) int32 rows of (s1, j1, s2, j2)."""
    a, b = _u8(a), _u8(b)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    n = a.shape[0] if r is None else r.shape[0]
    out = np.zeros((n, 4), np.int32)
    rc = _load().oracle_row_top2(_ptr(a), a.shape[0], _ptr(b), b.shape[0], _ptr(r), n, _ptr(out))
    assert rc == 0
    return out


def col_top2(a: np.ndarray, b: np.ndarray, cols=None) -> np.ndarray:
    """(n, 4) int32 columns of (c1, i1, c2, i2)."""
    a, b = _u8(a), _u8(b)
    c = None if cols is None else np.ascontiguousarray(cols, np.int32)
    n = b.shape[0] if c is None else c.shape[0]
    out = np.zeros((n, 4), np.int32)
    rc = _load().oracle_col_top2(_ptr(a), a.shape[0], _ptr(b), b.shape[0], _ptr(c), n, _ptr(out))
    assert rc == 0
    return out


def row_topk(a: np.ndarray, b: np.ndarray, k: int, rows=None):
    """Row top-k: (scores, index), each (n, k) int32, the first k candidates of every
    row (score descending, index ascending, zero scores excluded), padded (0, -1)."""
    a, b = _u8(a), _u8(b)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    n = a.shape[0] if r is None else r.shape[0]
    sc = np.zeros((n, max(k, 1)), np.int32)
    ix = np.zeros((n, max(k, 1)), np.int32)
    rc = _load().oracle_row_topk(_ptr(a), a.shape[0], _ptr(b), b.shape[0], int(k), _ptr(r), n, _ptr(sc), _ptr(ix))
    assert rc == 0, rc
    return sc, ix


@dataclass
class MatchResult:
    matches: np.ndarray   # (count, 2) int32, ascending i
    row_top2: np.ndarray  # (nA, 4)
    col_top2: np.ndarray  # (nB, 4)


def _capped(params: Params | None, n: int) -> int:
    k = (params or Params()).max_features
    return min(n, k) if k > 0 else n


def match(a: np.ndarray, b: np.ndarray, params: Params | None = None) -> MatchResult:
    """Whole-pair oracle: top-2 tables both ways and the match list (under a feature
    cap K the tables have min(n, K) rows)."""
    a, b = _u8(a), _u8(b)
    p = (params or Params())._c()
    na, nb = _capped(params, a.shape[0]), _capped(params, b.shape[0])
    rows = np.zeros((na, 4), np.int32)
    cols = np.zeros((nb, 4), np.int32)
    cap = max(na, 1)  # one match per row at most; min(nA, nB) only with the mutual check
    m = np.zeros((cap, 2), np.int32)
    cnt = np.zeros(1, np.int32)
    rc = _load().oracle_match(_ptr(a), a.shape[0], _ptr(b), b.shape[0], ctypes.byref(p), _ptr(rows),
                              _ptr(cols), _ptr(m), cap, _ptr(cnt))
    assert rc == 0
    return MatchResult(matches=m[: int(cnt[0])].copy(), row_top2=rows, col_top2=cols)


def accept_rows(a: np.ndarray, b: np.ndarray, rows, params: Params | None = None):
    """Sampled decisions: (j_or_minus1 (n,), row top-2 (n, 4), best column's top-2 (n, 4))."""
    a, b = _u8(a), _u8(b)
    p = (params or Params())._c()
    r = np.ascontiguousarray(rows, np.int32)
    n = r.shape[0]
    out_j = np.zeros(n, np.int32)
    out_r = np.zeros((n, 4), np.int32)
    out_c = np.zeros((n, 4), np.int32)
    rc = _load().oracle_accept_rows(_ptr(a), a.shape[0], _ptr(b), b.shape[0], ctypes.byref(p),
                                    _ptr(r), n, _ptr(out_j), _ptr(out_r), _ptr(out_c))
    assert rc == 0
    return out_j, out_r, out_c
