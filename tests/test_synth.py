"""The seeded input generators: determinism, shapes, value ranges, planted structure."""
import numpy as np

import sift_synth as S


def test_deterministic_and_shaped():
    p1 = S.single_pair_2000(0)
    p2 = S.single_pair_2000(0)
    assert p1.a.dtype == np.uint8 and p1.a.shape == (2000, 128) and p1.b.shape == (2000, 128)
    assert np.array_equal(p1.a, p2.a) and np.array_equal(p1.b, p2.b)
    assert np.array_equal(p1.truth, p2.truth)
    assert p1.truth.shape == (600, 2)
    assert len(set(p1.truth[:, 1].tolist())) == 600
    assert not np.array_equal(S.single_pair_2000(1).a, p1.a)


def test_sift_shape():
    p = S.single_pair_2000(0)
    sq = (p.a.astype(np.int64) ** 2).sum(1)
    assert sq.max() <= 512 * 512 and sq.min() > 0.9 * 512 * 512
    # clip at 0.2 -> no byte above floor(512 * 0.2 / min norm after clip) ~ 200s
    assert p.a.max() < 255


def test_planted_rows_are_close():
    p = S.single_pair_2000(0)
    i, j = p.truth[:, 0], p.truth[:, 1]
    d = np.abs(p.a[i].astype(np.int64) - p.b[j].astype(np.int64)).mean()
    other = np.abs(p.a[i].astype(np.int64) - p.b[(j + 1) % 2000].astype(np.int64)).mean()
    assert d < 0.6 * other


def test_ragged_sizes_range():
    s = S.ragged_sizes(0)
    assert s.shape == (256, 2) and s.min() >= 1000 and s.max() <= 16384
    p = S.ragged_pair(0, 3, s)
    assert p.a.shape[0] == s[3, 0] and p.b.shape[0] == s[3, 1]
    assert p.truth.shape[0] == int(0.15 * min(s[3]))


def test_ring_structure_small():
    r = S.make_ring(0, 77, 6, 400, 0.2, 0.06, 3)
    assert len(r.pairs) == 15
    k = 80
    for (i, j), t in r.truth.items():
        assert i < j and t.shape == (k, 2)
        assert len(set(t[:, 0].tolist())) == k
    # receivers' slots are disjoint across the three incoming sources
    recv = {}
    for (i, j), t in r.truth.items():
        d = (j - i) % 6
        rcv, col = (j, 1) if d in (1, 2, 3) else (i, 0)
        recv.setdefault(rcv, []).extend(t[:, col].tolist())
    for v in recv.values():
        assert len(v) == len(set(v))


def test_spot_pairs():
    s = S.survey_spot_pairs(0)
    assert s.shape == (50,) and len(set(s.tolist())) == 50 and s.max() < 4950
