"""Pins of the CPU oracle against things other than itself.

Each test names the mistakes it is there to catch:

* hand-worked examples (tests/golden/*.json, numbers derived by hand): dot product,
  zero floor and (0, -1) padding, lower-index tie-break both ways, strict ratio test,
  which side carries num and den, the gate's '>=', mutual check, column ratio test;
* an independent brute force (numpy int64 matmul, then a lexsort of every row and
  column) on tiny inputs with forced ties: transposed operands, index errors, a stale
  second-best, tie order, output order, empty and one-row inputs;
* planted-correspondence recovery on the seeded 2,000 x 2,000 workload (every planted
  row is recovered and nothing else is accepted);
* symmetry: match(B, A) is match(A, B) with i and j swapped when both directions run
  the same test;
* the bound s <= N = 512^2 on generated descriptors (Cauchy-Schwarz after floor
  quantisation);
* the derivation of the default parameters from 0.8 and 0.7 rad;
* row top-k: a hand-worked k = 6 example (ties in column order, zero floor, padding),
  a Python brute force on tiny inputs, k = 2 against the row top-2, and every k a
  prefix of k + 1.
"""
import json
import math
import os

import numpy as np
import pytest

import sift_synth as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _vec(spec):
    v = np.zeros(128, np.uint8)
    for d, x in spec:
        v[d] = x
    return v


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ hand-worked

def test_hand_4x4(oracle_mod):
    g = _load("hand_4x4.json")
    vec = {k: _vec(v) for k, v in g["vectors"].items()}
    A = np.stack([vec[k] for k in g["A"]])
    B = np.stack([vec[k] for k in g["B"]])
    assert oracle_mod.scores(A, B).tolist() == g["scores"]
    r = oracle_mod.match(A, B, oracle_mod.Params(col_ratio=1))
    assert r.row_top2.tolist() == g["row_top2"]
    assert r.col_top2.tolist() == g["col_top2"]
    assert r.matches.tolist() == g["matches_col_ratio_1"]
    r0 = oracle_mod.match(A, B, oracle_mod.Params(col_ratio=0))
    assert r0.matches.tolist() == g["matches_col_ratio_0"]
    # without the mutual check row 2 (best column 2, whose best row is 1) would pass
    r00 = oracle_mod.match(A, B, oracle_mod.Params(col_ratio=0, mutual=0))
    assert r00.matches.tolist() == [[1, 2], [2, 2]]


@pytest.mark.parametrize("case", ["tie", "pass"])
def test_ratio_boundary(oracle_mod, case):
    g = _load("ratio_boundary.json")
    A = np.stack([_vec(s) for s in g["A"]])
    B = np.stack([_vec(s) for s in g["B_" + case]])
    p = oracle_mod.Params(**g["params"])
    r = oracle_mod.match(A, B, p)
    assert r.row_top2[0].tolist() == g["row_top2_" + case]
    assert r.matches.tolist() == g["matches_" + case]


@pytest.mark.parametrize("case", ["at", "below"])
def test_gate_boundary(oracle_mod, case):
    g = _load("gate_boundary.json")
    A = np.stack([_vec(s) for s in g["A"]])
    B = np.stack([_vec(s) for s in g["B_" + case]])
    p = oracle_mod.default_params()
    assert p.min_score == g["min_score"]
    r = oracle_mod.match(A, B, p)
    assert r.row_top2[0].tolist() == [g["s_" + case], 0, 0, -1]
    assert r.matches.tolist() == g["matches_" + case]


@pytest.mark.parametrize("case", [0, 1, 2])
def test_feature_cap(oracle_mod, case):
    """SERAC page, 'Memory': the match cap clamps away the features past it.  The
    hand-worked capped 4x4 pair, and the cap against plain truncation of the inputs."""
    g = _load("feature_cap.json")
    c = g["cases"][case]
    vec = {k: _vec(v) for k, v in g["vectors"].items()}
    A = np.stack([vec[k] for k in g["A"]])
    B = np.stack([vec[k] for k in g["B"]])
    r = oracle_mod.match(A, B, oracle_mod.Params(col_ratio=1, max_features=c["max_features"]))
    assert r.row_top2.tolist() == c["row_top2"]
    assert r.col_top2.tolist() == c["col_top2"]
    assert r.matches.tolist() == c["matches_col_ratio_1"]
    r0 = oracle_mod.match(A, B, oracle_mod.Params(col_ratio=0, max_features=c["max_features"]))
    assert r0.matches.tolist() == c["matches_col_ratio_0"]


def test_feature_cap_is_truncation(oracle_mod):
    a, b = _tiny_inputs(11, 60, 45, 3)
    for k in (1, 7, 44, 45, 59, 200):
        p = oracle_mod.Params(norm_sq=60000, min_score=0, max_features=k)
        rows, cols, m = _brute(a[:k], b[:k], p)
        r = oracle_mod.match(a, b, p)
        assert r.row_top2.tolist() == rows and r.col_top2.tolist() == cols and r.matches.tolist() == m
        j, rr, _ = oracle_mod.accept_rows(a, b, np.arange(min(k, 60)), p)
        kept = {i: jj for i, jj in m}
        assert j.tolist() == [kept.get(i, -1) for i in range(min(k, 60))] and rr.tolist() == rows


def test_default_params(oracle_mod):
    p = oracle_mod.default_params(0.8, 0.7)
    assert (p.ratio_num_sq, p.ratio_den_sq) == (16, 25)
    # cos(0.7) * 2^18 = 200498.79...; far (0.21) from an integer, so double is enough
    x = math.cos(0.7) * 262144
    assert 200498.7 < x < 200498.8
    assert p.min_score == 200499 and p.norm_sq == 262144
    assert oracle_mod.default_params(1.0, 0.7).ratio_num_sq == oracle_mod.default_params(1.0, 0.7).ratio_den_sq


# ------------------------------------------------------------------ brute force

def _brute(a, b, p):
    """Independent restatement: full int64 matrix, then sort every row and column."""
    s = a.astype(np.int64) @ b.astype(np.int64).T
    na, nb = s.shape

    def top2(vals):
        idx = np.nonzero(vals > 0)[0]
        order = idx[np.lexsort((idx, -vals[idx]))]
        out = []
        for t in range(2):
            out += [int(vals[order[t]]), int(order[t])] if t < len(order) else [0, -1]
        return out

    rows = [top2(s[i]) for i in range(na)]
    cols = [top2(s[:, j]) for j in range(nb)]

    def ok(t):
        return t[1] >= 0 and p.ratio_den_sq * (p.norm_sq - t[0]) < p.ratio_num_sq * (p.norm_sq - t[2]) \
            and t[0] >= p.min_score

    m = []
    for i in range(na):
        t = rows[i]
        if not ok(t):
            continue
        c = cols[t[1]]
        if p.mutual and c[1] != i:
            continue
        if p.col_ratio and not ok(c):
            continue
        m.append([i, t[1]])
    return rows, cols, m


def _tiny_inputs(seed, na, nb, levels):
    """Small value alphabets and duplicated rows/columns force exact score ties."""
    rng = np.random.default_rng([seed, na, nb, levels])
    vals = np.array([0, 1, 2, 255] if levels == 4 else list(range(levels)), np.int64)
    a = vals[rng.integers(0, len(vals), size=(na, 128))].astype(np.uint8)
    b = vals[rng.integers(0, len(vals), size=(nb, 128))].astype(np.uint8)
    a[rng.random((na, 128)) < 0.6] = 0
    b[rng.random((nb, 128)) < 0.6] = 0
    if na > 2:
        a[na - 1] = a[0]
    if nb > 3:
        b[nb - 1] = b[1]
        b[2] = b[1]
    return a, b


@pytest.mark.parametrize("na,nb", [(0, 0), (0, 5), (5, 0), (1, 1), (1, 2), (2, 1), (2, 2),
                                   (3, 7), (17, 5), (33, 64), (64, 64), (64, 31)])
@pytest.mark.parametrize("levels", [2, 3, 4])
def test_brute_force_tiny(oracle_mod, na, nb, levels):
    a, b = _tiny_inputs(7, na, nb, levels)
    # a gate of 0 and a large N make the ratio test the deciding part on these inputs
    for p in [oracle_mod.Params(norm_sq=60000, min_score=0, col_ratio=1),
              oracle_mod.Params(norm_sq=60000, min_score=0, col_ratio=0),
              oracle_mod.Params(norm_sq=60000, min_score=0, mutual=0, col_ratio=0),
              oracle_mod.Params()]:
        rows, cols, m = _brute(a, b, p)
        r = oracle_mod.match(a, b, p)
        assert r.row_top2.tolist() == rows
        assert r.col_top2.tolist() == cols
        assert r.matches.tolist() == m


def test_brute_force_uniform_bytes(oracle_mod):
    a = S.random_u8(1, 40)
    b = S.random_u8(2, 50)
    p = oracle_mod.Params(norm_sq=4_000_000, min_score=0)
    rows, cols, m = _brute(a, b, p)
    r = oracle_mod.match(a, b, p)
    assert r.row_top2.tolist() == rows and r.col_top2.tolist() == cols and r.matches.tolist() == m


def test_sampled_entry_points_agree_with_brute_force(oracle_mod):
    a, b = _tiny_inputs(3, 48, 40, 3)
    p = oracle_mod.Params(norm_sq=60000, min_score=0)
    rows, cols, m = _brute(a, b, p)
    sel_r = np.array([0, 5, 47, 5], np.int32)
    sel_c = np.array([39, 0, 2], np.int32)
    assert oracle_mod.row_top2(a, b, sel_r).tolist() == [rows[i] for i in sel_r]
    assert oracle_mod.col_top2(a, b, sel_c).tolist() == [cols[j] for j in sel_c]
    j, rr, cc = oracle_mod.accept_rows(a, b, np.arange(48), p)
    kept = {i: jj for i, jj in m}
    assert j.tolist() == [kept.get(i, -1) for i in range(48)]
    assert rr.tolist() == rows


def test_scores_exact_extremes(oracle_mod):
    a = np.full((2, 128), 255, np.uint8)
    a[1, ::2] = 1
    b = np.full((3, 128), 255, np.uint8)
    b[1] = 0
    b[2, 0] = 1
    s = oracle_mod.scores(a, b)
    assert s[0, 0] == 128 * 255 * 255 == 8323200
    assert s[0, 1] == 0 and s[1, 0] == 64 * 255 + 64 * 255 * 255
    assert s[0, 2] == 127 * 255 * 255 + 255


# ------------------------------------------------------------------ planted truth

def test_planted_recovery_2000(oracle_mod):
    p = S.single_pair_2000(0)
    r = oracle_mod.match(p.a, p.b)
    truth = {tuple(x) for x in p.truth.tolist()}
    got = {tuple(x) for x in r.matches.tolist()}
    assert len(truth) == 600
    assert got == truth
    assert np.all(np.diff(r.matches[:, 0]) > 0)


def test_symmetry(oracle_mod):
    p = S.make_pair(5, 9, 0, 700, 500, 0.3, 0.05)
    ab = oracle_mod.match(p.a, p.b)
    ba = oracle_mod.match(p.b, p.a)
    assert np.array_equal(ab.row_top2, ba.col_top2)
    assert np.array_equal(ab.col_top2, ba.row_top2)
    swapped = ba.matches[:, ::-1]
    swapped = swapped[np.argsort(swapped[:, 0], kind="stable")]
    assert swapped.tolist() == ab.matches.tolist()


def test_score_bound_on_generated_data(oracle_mod):
    p = S.single_pair_2000(0)
    s = oracle_mod.scores(p.a[:300], p.b[:300])
    assert s.max() <= 512 * 512
    na = (p.a.astype(np.int64) ** 2).sum(1)
    assert na.max() <= 512 * 512


# ------------------------------------------------------------------ row top-k

def test_row_topk_hand(oracle_mod):
    g = _load("row_topk.json")
    vec = {k: _vec(v) for k, v in g["vectors"].items()}
    A = np.stack([vec[k] for k in g["A"]])
    B = np.stack([vec[k] for k in g["B"]])
    assert oracle_mod.scores(A, B).tolist() == g["scores"]
    sc, ix = oracle_mod.row_topk(A, B, g["k"])
    assert sc.tolist() == g["top_scores"]
    assert ix.tolist() == g["top_index"]
    for k in range(1, g["k"] + 1):   # every k is the first k columns of the k = 6 lists
        sk, ik = oracle_mod.row_topk(A, B, k)
        assert sk.tolist() == [r[:k] for r in g["top_scores"]]
        assert ik.tolist() == [r[:k] for r in g["top_index"]]


def _topk_brute(A, B, k):
    """Python loops: every candidate of the row, sorted by (-s, j), first k, padded."""
    out_s, out_j = [], []
    for i in range(A.shape[0]):
        cand = []
        for j in range(B.shape[0]):
            s = sum(int(x) * int(y) for x, y in zip(A[i], B[j]))
            if s > 0:
                cand.append((-s, j))
        cand.sort()
        cand = cand[:k] + [(0, -1)] * max(0, k - len(cand))
        out_s.append([-c[0] if c[1] >= 0 else 0 for c in cand])
        out_j.append([c[1] for c in cand])
    return out_s, out_j


@pytest.mark.parametrize("na,nb,k,seed", [(0, 5, 3, 0), (4, 0, 3, 1), (1, 1, 1, 2), (7, 9, 4, 3),
                                          (12, 10, 8, 4), (5, 3, 7, 5), (9, 16, 2, 6)])
def test_row_topk_brute_force(oracle_mod, na, nb, k, seed):
    rng = np.random.default_rng([seed, 77])
    # few distinct values so that ties are common, plus all-zero rows and columns
    A = rng.integers(0, 3, (na, 128)).astype(np.uint8) * rng.integers(0, 2, (na, 1)).astype(np.uint8)
    B = rng.integers(0, 3, (nb, 128)).astype(np.uint8)
    if nb > 2:
        B[1] = B[nb - 1]            # duplicated columns: equal scores, lower index first
        B[0] = 0
    bs, bj = _topk_brute(A, B, k)
    sc, ix = oracle_mod.row_topk(A, B, k)
    assert sc.tolist() == bs and ix.tolist() == bj


def test_row_topk_k2_is_row_top2(oracle_mod):
    p = S.single_pair_2000(0)
    a, b = p.a[:300], p.b[:700]
    b = np.concatenate([b, b[:50]])   # exact ties with lower columns
    sc, ix = oracle_mod.row_topk(a, b, 2)
    t2 = oracle_mod.row_top2(a, b)
    assert np.array_equal(np.stack([sc[:, 0], ix[:, 0], sc[:, 1], ix[:, 1]], 1), t2)


def test_row_topk_rows_and_arguments(oracle_mod):
    p = S.single_pair_2000(0)
    a, b = p.a[:64], p.b[:200]
    sc, ix = oracle_mod.row_topk(a, b, 5)
    rows = np.array([63, 0, 17, 17], np.int32)
    s2, i2 = oracle_mod.row_topk(a, b, 5, rows=rows)
    assert np.array_equal(s2, sc[rows]) and np.array_equal(i2, ix[rows])
    lib = oracle_mod._load()
    out = np.zeros((64, 1), np.int32)
    P = oracle_mod._ptr
    assert lib.oracle_row_topk(P(a), 64, P(b), 200, 0, None, 0, P(out), P(out)) == -1   # k < 1
    bad = np.array([64], np.int32)
    assert lib.oracle_row_topk(P(a), 64, P(b), 200, 1, P(bad), 1, P(out), P(out)) == -1  # row out of range
