"""GPU parity of the row top-k (guided matching) path against the CPU oracle, bit-exact.

Every entry (score and column) of every row is compared, on sizes that span several
tiles with ragged tails, on tie-heavy inputs (duplicated columns, zero rows and
columns), for every k the kernels serve (1..8, on both top-k builds), at the full
8192 x 8192 size on sampled rows, against the top-2 of match_pair for k = 2, and
through a timeout that the kernels report without a fault.
"""
import numpy as np
import pytest
import torch

import sift_synth as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def serac():
    import top_ratio_test_gb300 as s
    assert torch.cuda.is_available()
    assert s.device_check() == s.OK, s.status_str(s.device_check())
    return s


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _topk(serac, a, b, k, **kw):
    out = serac.topk_pair(_dev(a), _dev(b), k, **kw)
    torch.cuda.synchronize()
    assert int(out.status.item()) == serac.OK
    n = a.shape[0]
    return out.scores.cpu().numpy()[:n], out.index.cpu().numpy()[:n]


def _tie_pair(seed, na, nb):
    rng = np.random.default_rng([seed, 91])
    a = rng.integers(0, 4, (na, 128)).astype(np.uint8)
    b = rng.integers(0, 4, (nb, 128)).astype(np.uint8)
    if nb > 300:
        b[260:300] = b[5:45]          # equal scores in another tile, lower column first
        b[7] = b[3]                   # and in the same half
        b[40] = 0                     # a zero column
    if na > 10:
        a[9] = 0                      # a row with no candidate at all
    return a, b


@pytest.mark.parametrize("na,nb", [(1, 1), (129, 300), (700, 1031), (2000, 2000), (300, 4100)])
@pytest.mark.parametrize("k", [1, 4, 5, 8])
def test_topk_ragged(serac, oracle_mod, na, nb, k):
    p = S.make_pair(3, 7, na * 10 + nb, na, nb, 0.25, 0.08)
    sc, ix = _topk(serac, p.a, p.b, k)
    rs, ri = oracle_mod.row_topk(p.a, p.b, k)
    np.testing.assert_array_equal(sc, rs)
    np.testing.assert_array_equal(ix, ri)


@pytest.mark.parametrize("k", [2, 3, 6, 7])
def test_topk_ties(serac, oracle_mod, k):
    a, b = _tie_pair(k, 400, 1100)
    sc, ix = _topk(serac, a, b, k)
    rs, ri = oracle_mod.row_topk(a, b, k)
    np.testing.assert_array_equal(sc, rs)
    np.testing.assert_array_equal(ix, ri)


@pytest.mark.parametrize("na,nb,k", [(130, 20000, 3), (9000, 300, 8), (256, 65536, 1)])
def test_topk_extreme_aspect(serac, oracle_mod, na, nb, k):
    """Few row tiles against many column tiles: a row tile's columns are cut into dozens
    of pieces (one list slot each); many row tiles against one column tile: one slot."""
    p = S.make_pair(4, 7, na + nb, na, nb, 0.25, 0.08)
    sc, ix = _topk(serac, p.a, p.b, k)
    rows = np.unique(np.concatenate([np.arange(0, na, max(1, na // 64)), [na - 1]])).astype(np.int32)
    rs, ri = oracle_mod.row_topk(p.a, p.b, k, rows=rows)
    np.testing.assert_array_equal(sc[rows], rs)
    np.testing.assert_array_equal(ix[rows], ri)


def test_topk2_equals_row_top2(serac):
    p = S.single_pair_2000(0)
    sc, ix = _topk(serac, p.a, p.b, 2)
    out = serac.match_pair(_dev(p.a), _dev(p.b), top2=True)
    torch.cuda.synchronize()
    t2 = out.row_top2.cpu().numpy()
    np.testing.assert_array_equal(np.stack([sc[:, 0], ix[:, 0], sc[:, 1], ix[:, 1]], 1), t2)


def test_topk_8192_sampled(serac, oracle_mod):
    p = S.single_pair_8192(0)
    sc, ix = _topk(serac, p.a, p.b, 8)
    rows = np.random.default_rng(11).choice(8192, 96, replace=False).astype(np.int32)
    rows = np.concatenate([rows, np.array([0, 127, 128, 8191], np.int32)])
    rs, ri = oracle_mod.row_topk(p.a, p.b, 8, rows=rows)
    np.testing.assert_array_equal(sc[rows], rs)
    np.testing.assert_array_equal(ix[rows], ri)
    # every row: descending scores, positive scores with valid distinct columns, then (0, -1)
    assert np.all(np.diff(sc.astype(np.int64), axis=1) <= 0)
    assert np.all((sc > 0) == (ix >= 0)) and np.all(ix < 8192)


def test_topk_empty_sides(serac, oracle_mod):
    p = S.make_pair(5, 7, 1, 300, 300, 0.25, 0.08)
    sc, ix = _topk(serac, p.a, p.b[:0], 3)        # no columns: every row is padding
    assert sc.tolist() == [[0, 0, 0]] * 300 and ix.tolist() == [[-1, -1, -1]] * 300
    out = serac.topk_pair(_dev(p.a[:0]), _dev(p.b), 3)   # no rows: nothing to write
    torch.cuda.synchronize()
    assert int(out.status.item()) == serac.OK


def test_topk_host_outputs_and_reuse(serac, oracle_mod):
    p = S.make_pair(6, 7, 2, 900, 1300, 0.25, 0.08)
    ws = serac.workspace(serac.topk_workspace_size(900, 1300, 6), torch.device("cuda", 0))
    out = serac.topk_pair(_dev(p.a), _dev(p.b), 6, workspace_t=ws, host_out=True)
    torch.cuda.synchronize()
    rs, ri = oracle_mod.row_topk(p.a, p.b, 6)
    np.testing.assert_array_equal(out.scores.numpy(), rs)
    np.testing.assert_array_equal(out.index.numpy(), ri)
    q = S.make_pair(6, 8, 2, 900, 1300, 0.25, 0.08)   # same buffers and workspace, other data
    serac.topk_pair(_dev(q.a), _dev(q.b), 6, workspace_t=ws, out=out)
    torch.cuda.synchronize()
    rs, ri = oracle_mod.row_topk(q.a, q.b, 6)
    np.testing.assert_array_equal(out.scores.numpy(), rs)
    np.testing.assert_array_equal(out.index.numpy(), ri)


def test_topk_workspace_checks(serac):
    a = torch.zeros((300, 128), dtype=torch.uint8, device="cuda")
    need = serac.topk_workspace_size(300, 300, 4)
    assert need > 0
    with pytest.raises(serac.SeracError) as ei:
        serac.topk_pair(a, a, 4, workspace_t=serac.workspace(need - 1024, a.device))
    assert ei.value.status == serac.EWORKSPACE


def test_topk_timeout_is_reported(serac, oracle_mod):
    p = S.make_pair(7, 7, 3, 500, 700, 0.25, 0.08)
    serac.inject_timeout(True)
    out = serac.topk_pair(_dev(p.a), _dev(p.b), 4)
    torch.cuda.synchronize()
    assert int(out.status.item()) == serac.ETIMEOUT
    sc, ix = _topk(serac, p.a, p.b, 4)              # the next call is exact again
    rs, ri = oracle_mod.row_topk(p.a, p.b, 4)
    np.testing.assert_array_equal(sc, rs)
    np.testing.assert_array_equal(ix, ri)
