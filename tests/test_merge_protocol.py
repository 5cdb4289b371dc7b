"""Host simulation of the fused kernel's order-independent top-2 merge rules (CPU).

The fused kernel never sees a row whole: it reaches each row's top-2 through merge
steps whose order depends on which CTA or atomic happens to run first.  "Real-Time
Dense Stereo at 34 Hz on a Jetson TX2 (MASDA, Part 3)", section 6, checks its fused
warp top-2 the same way: a host simulation of the exact reduction must give the
sequential scan's result.  Here the kernel's rules are restated in numpy, driven
under many random and adversarial orders (exact ties, s = 0, the largest score
8,323,200, duplicated rows and columns), and compared with the sequential scan: the
oracle's row_top2 / col_top2, or a sort.

Every pair is matched as two row problems: the rows of A against the columns B, and
the rows of B against the columns A, whose row top-2 is the pair's column top-2.  A
problem is cut into 128 x 256 tiles; a thread holds one row of a tile and reads 64 of
its columns (a quarter) at once.  The rules, as the kernel applies them:

  K  32-bit tile keys s << 8 | (255 - index in the tile), compared as IEEE floats
     (max, min and the 3-input max): every key is below 0x7F800000, so the float
     order is the integer order, denormal keys (s < 2^15) included.
  T  a thread's top-2 of each 32-column half by a pairwise min/max tree over keys
     with a 5-bit index (31 - k), then the two halves merged with their upper index
     bits OR-ed in.
  F  the fold over a segment's tiles in column order: a tile key displaces a held one
     only when k > (R | 255) (a strictly larger score).
  A  the global top-2 by three atomicMax at the end of a segment: old = max(best,
     x1); max(second, x2); later max(second, min(old, x1)).  (Optionally gated: a
     contributor whose x1 does not exceed a past value of `second` skips all three,
     which the protocol also allows.)
"""
import numpy as np
import pytest

U32 = np.uint32
U64 = np.uint64
BM, BN = 128, 256


# ------------------------------------------------------------------ the rules

def fmax(a, b):
    return np.maximum(a.view(np.float32), b.view(np.float32)).view(U32)


def fmin(a, b):
    return np.minimum(a.view(np.float32), b.view(np.float32)).view(U32)


def merge2(a1, a2, b1, b2):
    """Top-2 (a1, a2) merged with (b1, b2): min, max, 3-input max (rule K)."""
    m = fmin(a1, b1)
    return fmax(a1, b1), fmax(fmax(a2, m), b2)


def tree_top2(x):
    """Rule T on the last axis: pairwise max/min, then pairwise merges."""
    hi = fmax(x[..., 0::2], x[..., 1::2])
    lo = fmin(x[..., 0::2], x[..., 1::2])
    while hi.shape[-1] > 1:
        hi, lo = merge2(hi[..., 0::2], lo[..., 0::2], hi[..., 1::2], lo[..., 1::2])
    return hi[..., 0], lo[..., 0]


def raw(s):
    """Accumulator bits of 2^23 + s: the integer 0x4B000000 | s."""
    return (U32(0x4B000000) | np.asarray(s).astype(U32)).astype(U32)


def half_bits(qt, c):
    """Rule T: the upper index bits of half c of quarter qt."""
    return U32((7 - 2 * qt - c) << 5)


def quarter_top2(s64, qt):
    """Rules K and T: a thread's top-2 over its 64 columns of quarter qt, as tile keys
    with index 255 - (64 qt + 32 c + k)."""
    v = raw(s64)
    t1 = np.zeros(s64.shape[:-1], U32)
    t2 = np.zeros(s64.shape[:-1], U32)
    for c in range(2):
        keys = (v[..., 32 * c:32 * c + 32] * U32(256) + (U32(31) - np.arange(32, dtype=U32))).astype(U32)
        a1, a2 = tree_top2(keys)
        b = half_bits(qt, c)
        t1, t2 = merge2(t1, t2, a1 | b, a2 | b)
    return t1, t2


def fold(R1, C1, R2, C2, k1t, k2t, ct):
    """Rule F for one tile of column-tile index ct (vectorised over rows)."""
    enter = k1t > (R2 | U32(255))
    top = enter & (k1t > (R1 | U32(255)))
    t2_wins = k2t > (R1 | U32(255))
    nR2 = np.where(top, np.where(t2_wins, k2t, R1), np.where(enter, k1t, R2)).astype(U32)
    nC2 = np.where(top, np.where(t2_wins, ct, C1), np.where(enter, ct, C2))
    return np.where(top, k1t, R1).astype(U32), np.where(top, ct, C1), nR2, nC2


def key64(k, base):
    """32-bit tile keys -> 64-bit s << 32 | ~(base + index); 0 when s == 0."""
    k = np.asarray(k).astype(U64)
    s = k >> U64(8)
    idx = np.asarray(base).astype(U64) + (U64(255) - (k & U64(255)))
    return np.where(s == 0, U64(0), (s << U64(32)) | (U64(0xFFFFFFFF) - idx))


def decode(best, second):
    def one(k):
        s = (k >> U64(32)).astype(np.int64)
        i = np.where(k == 0, -1, (U64(0xFFFFFFFF) - (k & U64(0xFFFFFFFF))).astype(np.int64))
        return s, i
    s1, i1 = one(best)
    s2, i2 = one(second)
    return np.stack([s1, i1, s2, i2], axis=-1).astype(np.int64)


class Global:
    """Global (best, second) 64-bit keys of rows, updated by rule A with contributions
    that arrive in an arbitrary order."""

    def __init__(self, n):
        self.best = np.zeros(n, U64)
        self.second = np.zeros(n, U64)

    def run(self, contribs, rng, gate=False):
        """contribs: list of (index, x1, x2).  Each contributor's three atomics happen
        at random times (the deferred min after its first); with `gate`, it first reads
        `second` at a random earlier time and skips everything if x1 does not exceed it."""
        events = []
        for c in range(len(contribs)):
            t_read = rng.random()
            t1 = t_read + rng.random()
            events += [(t_read, 0, c), (t1, 1, c), (t1 + 0.5 * rng.random(), 2, c), (t1 + rng.random(), 3, c)]
        events.sort()
        seen, old = {}, {}
        for _, kind, c in events:
            j, x1, x2 = contribs[c]
            if kind == 0:
                seen[c] = self.second[j] if gate else U64(0)
            elif not x1 or x1 <= seen[c]:
                continue
            elif kind == 1:
                old[c] = self.best[j]
                self.best[j] = max(self.best[j], x1)
            elif kind == 2:
                if x2:
                    self.second[j] = max(self.second[j], x2)
            else:
                lo = min(old[c], x1)
                if lo:
                    self.second[j] = max(self.second[j], lo)


# ------------------------------------------------------------------ rule tests

def _scores(rng, shape):
    """Scores with many exact ties, zeros, denormal-key values and the largest score."""
    pool = np.array([0, 0, 1, 2, 3, 255, 32767, 32768, 65025, 200499, 262144, 8323199, 8323200], np.int64)
    s = pool[rng.integers(0, len(pool), size=shape)]
    mix = rng.random(shape) < 0.3
    s[mix] = rng.integers(0, 8323201, size=int(mix.sum()))
    return s


def test_tree_top2_equals_sort():
    """Rules K and T: 200,000 halves of 32 keys (distinct index bits)."""
    rng = np.random.default_rng(1)
    keys = (raw(_scores(rng, (200_000, 32))) * U32(256) + (U32(31) - np.arange(32, dtype=U32))).astype(U32)
    k1, k2 = tree_top2(keys)
    srt = np.sort(keys, axis=-1)
    assert np.array_equal(k1, srt[:, -1]) and np.array_equal(k2, srt[:, -2])
    assert keys.max() < 0x7F800000  # float order is the integer order for every key


@pytest.mark.parametrize("qt", [0, 1, 2, 3])
def test_quarter_top2_equals_sort(qt):
    """Rules K and T over a thread's 64 columns (two halves), 100,000 rows."""
    rng = np.random.default_rng([2, qt])
    s = _scores(rng, (100_000, 64))
    t1, t2 = quarter_top2(s, qt)
    keys = (raw(s) * U32(256) + (U32(255) - U32(64 * qt) - np.arange(64, dtype=U32))).astype(U32)
    srt = np.sort(keys, axis=-1)
    assert np.array_equal(t1, srt[:, -1]) and np.array_equal(t2, srt[:, -2])


def _scan(row):
    """Sequential scan: top-2 of (score, index) with the zero floor, lower index first."""
    idx = np.nonzero(row > 0)[0]
    o = idx[np.lexsort((idx, -row[idx]))]
    return [int(row[o[0]]) if len(o) else 0, int(o[0]) if len(o) else -1,
            int(row[o[1]]) if len(o) > 1 else 0, int(o[1]) if len(o) > 1 else -1]


def test_fold_equals_sequential_scan():
    """Rule F: 20,000 rows over 1..12 tiles (one quarter of 64 columns each), whole
    tiles repeated so that ties meet across tiles; the segment's top-2 equals the scan."""
    rng = np.random.default_rng(3)
    n, tiles = 20_000, 12
    s = _scores(rng, (n, tiles, 64))
    s[rng.random((n, tiles, 64)) < 0.2] = 0
    dup = rng.random(n) < 0.3
    s[dup, 5] = s[dup, 2]
    s[dup, 7, :32] = s[dup, 3, 32:]            # equal scores at a lower index in a later tile
    length = rng.integers(1, tiles + 1, size=n)
    R1, R2 = np.zeros(n, U32), np.zeros(n, U32)
    C1, C2 = np.zeros(n, np.int64), np.zeros(n, np.int64)
    for ct in range(tiles):
        k1t, k2t = quarter_top2(s[:, ct], 0)
        nxt = fold(R1, C1, R2, C2, k1t, k2t, ct)
        live = ct < length
        R1, C1, R2, C2 = (np.where(live, a, b) for a, b in zip(nxt, (R1, C1, R2, C2)))
    got = decode(key64(R1, 64 * C1), key64(R2, 64 * C2))
    for i in range(n):
        assert got[i].tolist() == _scan(s[i, :length[i]].reshape(-1)), i


@pytest.mark.parametrize("gate", [False, True])
def test_atomic_top2_any_order(gate):
    """Rule A: 100,000 trials of up to 8 contributors (disjoint column sets, so keys are
    unique) in random orders: the final (best, second) is the top-2 of all keys."""
    rng = np.random.default_rng([5, gate])
    trials = 100_000
    g = Global(trials)
    contribs, expect = [], np.zeros((trials, 2), U64)
    for t in range(trials):
        k = int(rng.integers(1, 9))
        s = np.sort(_scores(rng, (k, 2)), axis=1)
        cols = rng.permutation(64)[:2 * k].reshape(k, 2)
        keys = []
        for c in range(k):
            pair = sorted([(U64(int(s[c, 1])) << U64(32)) | U64(0xFFFFFFFF - int(cols[c, 0])) if s[c, 1] else U64(0),
                           (U64(int(s[c, 0])) << U64(32)) | U64(0xFFFFFFFF - int(cols[c, 1])) if s[c, 0] else U64(0)])
            contribs.append((t, pair[1], pair[0]))
            keys += pair
        srt = sorted(keys)
        expect[t] = [srt[-1], srt[-2]]
    g.run([contribs[i] for i in rng.permutation(len(contribs))], rng, gate=gate)
    assert np.array_equal(g.best, expect[:, 0]) and np.array_equal(g.second, expect[:, 1])


# ------------------------------------------------------------------ the whole kernel

def _simulate_problem(scores, grid, rng):
    """The fused kernel's reduction of one row problem, replayed on the host: 128 x 256
    tiles dealt to `grid` CTAs as contiguous row-major pieces and processed in steps
    (one tile per CTA per step, CTAs in a random order); a segment (a piece's run of
    tiles on one row tile) folds its tiles per row and quarter and flushes them through
    rule A, whose atomics arrive in a random order.  Returns the row top-2 (n, 4)."""
    na, nb = scores.shape
    rt_n, ct_n = -(-na // BM), -(-nb // BN)
    pad = np.zeros((rt_n * BM, ct_n * BN), np.int64)
    pad[:na, :nb] = scores
    q, r = divmod(rt_n * ct_n, grid)
    pieces = [(k * q + min(k, r), (k + 1) * q + min(k + 1, r)) for k in range(grid)]
    rows = Global(rt_n * BM)
    seg = {}
    for tau in range(max(e - s for s, e in pieces)):
        contribs = []
        for k in rng.permutation(grid):
            t = pieces[k][0] + tau
            if t >= pieces[k][1]:
                continue
            rt, ct = divmod(t, ct_n)
            if tau == 0 or ct == 0:
                seg[k] = [np.zeros((BM, 4), U32), np.zeros((BM, 4), np.int64),
                          np.zeros((BM, 4), U32), np.zeros((BM, 4), np.int64)]
            st = seg[k]
            blk = pad[rt * BM:(rt + 1) * BM, ct * BN:(ct + 1) * BN]
            for qt in range(4):
                t1, t2 = quarter_top2(blk[:, 64 * qt:64 * qt + 64], qt)
                st[0][:, qt], st[1][:, qt], st[2][:, qt], st[3][:, qt] = fold(
                    st[0][:, qt], st[1][:, qt], st[2][:, qt], st[3][:, qt], t1, t2, ct)
            if ct == ct_n - 1 or t + 1 == pieces[k][1]:
                K1, K2 = key64(st[0], BN * st[1]), key64(st[2], BN * st[3])
                for i in range(min(BM, na - rt * BM)):
                    for qt in range(4):
                        if K1[i, qt]:
                            contribs.append((rt * BM + i, K1[i, qt], K2[i, qt]))
        rows.run(contribs, rng)
    return decode(rows.best, rows.second)[:na]


def _tie_pair(rng, na, nb):
    vals = np.array([0, 1, 2, 255], np.uint8)
    a = vals[rng.integers(0, 4, size=(na, 128))]
    b = vals[rng.integers(0, 4, size=(nb, 128))]
    a[rng.random(a.shape) < 0.7] = 0
    b[rng.random(b.shape) < 0.7] = 0
    a[na // 3: na // 3 + 9] = a[1]               # repeated rows: ties in every column
    b[nb // 2: nb // 2 + 20] = b[3]              # repeated columns: ties in every row
    if nb > 300:
        b[40] = 255                              # the largest score in every row that has it ...
        b[256:276] = b[40]                       # ... tied in a later tile at lower in-tile indices
    if na > 300:
        a[100] = 255                             # the same for columns, across row tiles
        a[256:270] = a[100]
    a[0] = 255
    b[nb - 1] = 255
    a[2] = 0                                     # an all-zero row
    small = np.array([0, 1, 2], np.uint8)        # rows and columns whose best scores give
    a[3:8] = small[rng.integers(0, 3, size=(5, 128))]   # denormal keys (s < 2^15)
    a[3:8, rng.random(128) < 0.5] = 0
    b[5:9] = small[rng.integers(0, 3, size=(4, 128))]
    return a, b


@pytest.mark.parametrize("case", range(6))
def test_whole_kernel_simulation_equals_oracle(oracle_mod, case):
    """The host replay of both row problems of a pair equals the oracle's sequential
    scan, rows and columns, on pairs built for ties, over CTA counts that split rows
    among many contributors."""
    rng = np.random.default_rng([6, case])
    na, nb = [(300, 600), (129, 257), (400, 513), (128, 1100), (600, 256), (40, 70)][case]
    a, b = _tie_pair(rng, na, nb)
    sc = oracle_mod.scores(a, b).astype(np.int64)
    ref_r, ref_c = oracle_mod.row_top2(a, b), oracle_mod.col_top2(a, b)
    for grid in (1, 3, 7):
        assert np.array_equal(_simulate_problem(sc, grid, rng), ref_r), (case, grid)
        assert np.array_equal(_simulate_problem(sc.T.copy(), grid, rng), ref_c), (case, grid)


def test_simulation_catches_planted_mistakes(oracle_mod):
    """The replay is sharp enough to see a plausible slip in each rule: every planted
    mistake (in this simulation, never in the kernel) breaks the equality."""
    g = globals()
    good = {k: g[k] for k in ("fold", "half_bits", "fmax", "fmin")}
    good_run = Global.run

    def fold_plain(R1, C1, R2, C2, k1t, k2t, ct):       # F without the '| 255': later tiles win ties
        enter = k1t > R2
        top = enter & (k1t > R1)
        nR2 = np.where(top, np.where(k2t > R1, k2t, R1), np.where(enter, k1t, R2)).astype(U32)
        nC2 = np.where(top, np.where(k2t > R1, ct, C1), np.where(enter, ct, C2))
        return np.where(top, k1t, R1).astype(U32), np.where(top, ct, C1), nR2, nC2

    def half_bits_swapped(qt, c):                       # T: the halves' index bits swapped
        return U32((7 - 2 * qt - (1 - c)) << 5)

    def ftz(x):                                         # K: denormal keys flushed to zero, as a
        return np.where(x < U32(0x00800000), U32(0), x)  # build with -ftz=true would compare them

    def fmax_ftz(a, b):
        return np.maximum(ftz(a).view(np.float32), ftz(b).view(np.float32)).view(U32)

    def fmin_ftz(a, b):
        return np.minimum(ftz(a).view(np.float32), ftz(b).view(np.float32)).view(U32)

    def run_no_deferred(self, contribs, rng, gate=False):   # A without max(second, min(old, x1))
        for j, x1, x2 in contribs:
            self.best[j] = max(self.best[j], x1)
            if x2:
                self.second[j] = max(self.second[j], x2)

    rng = np.random.default_rng(7)
    a, b = _tie_pair(rng, 400, 600)
    sc = oracle_mod.scores(a, b).astype(np.int64)
    ref_r, ref_c = oracle_mod.row_top2(a, b), oracle_mod.col_top2(a, b)
    try:
        for name, fn in [("fold", fold_plain), ("half_bits", half_bits_swapped), ("ftz", (fmax_ftz, fmin_ftz)),
                         ("atomic", run_no_deferred)]:
            g.update(good)
            Global.run = good_run
            if name == "atomic":
                Global.run = fn
            elif name == "ftz":
                g["fmax"], g["fmin"] = fn
            else:
                g[name] = fn
            caught = False
            for grid in (1, 3, 7):
                caught |= not np.array_equal(_simulate_problem(sc, grid, rng), ref_r)
                caught |= not np.array_equal(_simulate_problem(sc.T.copy(), grid, rng), ref_c)
            assert caught, name
    finally:
        g.update(good)
        Global.run = good_run
