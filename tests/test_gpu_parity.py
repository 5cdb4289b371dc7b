"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit-exact.

Integer work, so the bar is equality everywhere: scores, row and column top-2
(score and index), and match lists (order included).
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


def _run_pair(serac, a, b, params=None, capacity=None):
    out = serac.match_pair(_dev(a), _dev(b), params, capacity=capacity, top2=True)
    torch.cuda.synchronize()
    return out


def _oracle_params(oracle_mod, p):
    return oracle_mod.Params(p.ratio_num_sq, p.ratio_den_sq, p.norm_sq, p.min_score, p.mutual, p.col_ratio,
                             p.max_features)


def _assert_pair(serac, oracle_mod, a, b, params=None):
    p = params if params is not None else serac.default_params()
    out = _run_pair(serac, a, b, p)
    ref = oracle_mod.match(a, b, _oracle_params(oracle_mod, p))
    na, nb = ref.row_top2.shape[0], ref.col_top2.shape[0]
    np.testing.assert_array_equal(out.row_top2.cpu().numpy()[:na], ref.row_top2)
    np.testing.assert_array_equal(out.col_top2.cpu().numpy()[:nb], ref.col_top2)
    np.testing.assert_array_equal(out.result().numpy(), ref.matches)
    return out, ref


# ------------------------------------------------------------------ contraction

def _adversarial(seed, na, nb):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 256, size=(na, 128)).astype(np.uint8)
    b = rng.integers(0, 256, size=(nb, 128)).astype(np.uint8)
    a[0] = 255                      # 8,323,200 against an all-255 row: the largest score
    b[0] = 255
    if na > 2:
        a[1] = 0
        a[1, 0] = 255               # one 255^2 product among zeros
        a[2, ::2] = 255
        a[2, 1::2] = 1
    if nb > 2:
        b[2] = 1                    # many 1 x k products
    return a, b


@pytest.mark.parametrize("na,nb", [(1, 1), (3, 300), (130, 257), (256, 512), (300, 700)])
def test_scores_exact(serac, oracle_mod, na, nb):
    a, b = _adversarial(na * 1000 + nb, na, nb)
    s = serac.scores(_dev(a), _dev(b))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s.cpu().numpy(), oracle_mod.scores(a, b))


def test_fused_equals_unfused(serac, oracle_mod):
    """Top-2 taken from the written-out score matrix equals the fused result."""
    a, b = _adversarial(5, 200, 600)
    a[10:20] = a[0]                 # duplicated rows and columns force ties
    b[30:40] = b[3]
    s = serac.scores(_dev(a), _dev(b)).cpu().numpy().astype(np.int64)
    out = _run_pair(serac, a, b)

    def top2(v):
        idx = np.nonzero(v > 0)[0]
        o = idx[np.lexsort((idx, -v[idx]))]
        return [int(v[o[0]]) if len(o) else 0, int(o[0]) if len(o) else -1,
                int(v[o[1]]) if len(o) > 1 else 0, int(o[1]) if len(o) > 1 else -1]

    assert out.row_top2.cpu().numpy().tolist() == [top2(s[i]) for i in range(200)]
    assert out.col_top2.cpu().numpy().tolist() == [top2(s[:, j]) for j in range(600)]


# ------------------------------------------------------------------ single pairs

def test_pair_2000(serac, oracle_mod):
    p = S.single_pair_2000(0)
    out, ref = _assert_pair(serac, oracle_mod, p.a, p.b)
    got = {tuple(x) for x in out.result().numpy().tolist()}
    assert got == {tuple(x) for x in p.truth.tolist()}


def test_pair_8192(serac, oracle_mod):
    p = S.single_pair_8192(0)
    out, ref = _assert_pair(serac, oracle_mod, p.a, p.b)
    assert len(ref.matches) > 1500


@pytest.mark.parametrize("na,nb", [(0, 0), (0, 7), (7, 0), (1, 1), (1, 300), (127, 129), (128, 256),
                                   (129, 255), (255, 257), (257, 1), (1000, 2300), (3001, 513)])
def test_ragged_sizes(serac, oracle_mod, na, nb):
    p = S.make_pair(1, 60, na * 7 + nb, na, nb, 0.3, 0.05)
    _assert_pair(serac, oracle_mod, p.a, p.b)


def test_largest_size(serac, oracle_mod):
    p = S.make_pair(2, 61, 0, 16384, 16384, 0.15, 0.05)
    _assert_pair(serac, oracle_mod, p.a, p.b)


@pytest.mark.parametrize("na,nb", [(128, 65536), (100, 40000), (65536, 200), (40000, 130)])
def test_extreme_aspect(serac, oracle_mod, na, nb):
    """One row tile against hundreds of column tiles (the row tile split over many CTAs,
    rows merged across them), and the reverse (hundreds of row tiles, one column tile:
    every column merged from hundreds of CTAs)."""
    p = S.make_pair(4, 63, na + nb, na, nb, 0.3, 0.05)
    _assert_pair(serac, oracle_mod, p.a, p.b)


def test_zero_and_identical_images(serac, oracle_mod):
    """All-zero descriptors score 0 everywhere (no candidate, no match); an image
    matched against itself has exact ties wherever rows repeat."""
    z = np.zeros((300, 128), np.uint8)
    p = S.make_pair(5, 64, 0, 700, 10, 0.0, 0.05)
    a = p.a.copy()
    a[100:140] = a[5]                     # 41 identical rows
    out, ref = _assert_pair(serac, oracle_mod, z, a)
    assert len(ref.matches) == 0 and (out.row_top2.cpu().numpy() == [0, -1, 0, -1]).all()
    _assert_pair(serac, oracle_mod, a, z)
    _assert_pair(serac, oracle_mod, a, a)


def test_batch_many_images_and_chunks(serac, oracle_mod):
    """300 pairs of 600 distinct small images: two staging launches (512 images each at
    most) and three launch chunks alternating between the two key regions."""
    pairs_np = [S.make_pair(6, 65, k, 40 + (k * 37) % 300, 30 + (k * 53) % 290, 0.3, 0.05) for k in range(300)]
    dev = [(_dev(p.a), _dev(p.b)) for p in pairs_np]
    outs = serac.match_batch(dev, top2=True)
    torch.cuda.synchronize()
    for k, p in enumerate(pairs_np):
        ref = oracle_mod.match(p.a, p.b)
        np.testing.assert_array_equal(outs[k].row_top2.cpu().numpy()[:p.a.shape[0]], ref.row_top2)
        np.testing.assert_array_equal(outs[k].col_top2.cpu().numpy()[:p.b.shape[0]], ref.col_top2)
        np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)


def test_batch_mixed_piece_sizes(serac, oracle_mod):
    """One launch chunk whose pairs are dealt across the CTAs in pieces of every kind:
    pairs with more tiles than CTAs and a remainder (480 and 213 tiles), one-tile
    pairs that each go to a single CTA, an empty pair, and a pair of 40 tiles, so the
    CTA offsets of the pieces rotate through the grid."""
    sizes = [(3000, 5000)] + [(100 + k, 90 + 3 * k) for k in range(20)] + [(0, 50), (2500, 300), (9000, 700)]
    pairs_np = [S.make_pair(7, 66, k, max(na, 1), nb, 0.2, 0.05) for k, (na, nb) in enumerate(sizes)]
    a_list = [p.a[:na] for p, (na, _) in zip(pairs_np, sizes)]
    b_list = [p.b for p in pairs_np]
    dev = [(_dev(a), _dev(b)) for a, b in zip(a_list, b_list)]
    outs = serac.match_batch(dev, top2=True)
    torch.cuda.synchronize()
    for k in range(len(sizes)):
        a, b = a_list[k], b_list[k]
        ref = oracle_mod.match(a, b)
        np.testing.assert_array_equal(outs[k].row_top2.cpu().numpy()[:a.shape[0]], ref.row_top2)
        np.testing.assert_array_equal(outs[k].col_top2.cpu().numpy()[:b.shape[0]], ref.col_top2)
        np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)


@pytest.mark.parametrize("variant", ["default", "no_col_ratio", "no_mutual", "loose"])
def test_ties_and_params(serac, oracle_mod, variant):
    rng = np.random.default_rng(11)
    vals = np.array([0, 1, 2, 255], np.uint8)
    a = vals[rng.integers(0, 4, size=(300, 128))]
    b = vals[rng.integers(0, 4, size=(500, 128))]
    a[rng.random(a.shape) < 0.7] = 0
    b[rng.random(b.shape) < 0.7] = 0
    a[150:160] = a[3]
    b[200:230] = b[7]
    b[499] = b[7]
    p = serac.default_params()
    if variant == "no_col_ratio":
        p.col_ratio = 0
    elif variant == "no_mutual":
        p.mutual, p.col_ratio = 0, 0
    elif variant == "loose":
        p.norm_sq, p.min_score = 2_000_000, 0
    _assert_pair(serac, oracle_mod, a, b, p)


def test_capacity_overflow_and_repeat(serac, oracle_mod):
    p = S.single_pair_2000(0)
    ref = oracle_mod.match(p.a, p.b)
    out = _run_pair(serac, p.a, p.b, capacity=100)
    assert int(out.count.item()) == len(ref.matches)
    np.testing.assert_array_equal(out.matches[:100].cpu().numpy(), ref.matches[:100])
    with pytest.raises(serac.SeracError):
        out.result()
    # same inputs twice on one workspace: identical
    a, b = _dev(p.a), _dev(p.b)
    ws = serac.workspace(serac.pair_workspace_size(2000, 2000), a.device)
    r1 = serac.match_pair(a, b, workspace_t=ws, top2=True)
    r2 = serac.match_pair(a, b, workspace_t=ws, top2=True)
    torch.cuda.synchronize()
    assert torch.equal(r1.row_top2, r2.row_top2) and torch.equal(r1.col_top2, r2.col_top2)
    assert torch.equal(r1.result(), r2.result())


def test_pinned_host_inputs_and_outputs(serac, oracle_mod):
    """Descriptors in pinned host memory (read by the staging kernel over the host link)
    and outputs written straight into pinned host memory give the same results."""
    p = S.make_pair(6, 64, 0, 1500, 1800, 0.3, 0.05)
    a = torch.from_numpy(p.a).pin_memory()
    b = torch.from_numpy(p.b).pin_memory()
    out = serac.match_pair(a, b, host_out=True, top2=True)
    got = out.result().numpy()
    ref = oracle_mod.match(p.a, p.b)
    assert not out.count.is_cuda
    np.testing.assert_array_equal(got, ref.matches)
    np.testing.assert_array_equal(out.row_top2.numpy(), ref.row_top2)
    np.testing.assert_array_equal(out.col_top2.numpy(), ref.col_top2)


def test_workspace_too_small(serac):
    a = torch.zeros((10, 128), dtype=torch.uint8, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(serac.SeracError) as e:
        serac.match_pair(a, a, workspace_t=ws)
    assert e.value.status == serac.EWORKSPACE


def test_same_image_both_sides(serac, oracle_mod):
    p = S.make_pair(3, 62, 0, 700, 10, 0.0, 0.05)
    a = _dev(p.a)
    out = serac.match_pair(a, a, top2=True)
    torch.cuda.synchronize()
    ref = oracle_mod.match(p.a, p.a)
    np.testing.assert_array_equal(out.row_top2.cpu().numpy(), ref.row_top2)
    np.testing.assert_array_equal(out.result().numpy(), ref.matches)


# ------------------------------------------------------------------ batches

def test_batch_ring_12(serac, oracle_mod):
    """12 images x 8,192, all 66 pairs through match_batch, every pair in full."""
    r = S.ring_12x8192(0)
    imgs = [_dev(x) for x in r.images]
    outs = serac.match_batch([(imgs[i], imgs[j]) for i, j in r.pairs], top2=True)
    torch.cuda.synchronize()
    for k, (i, j) in enumerate(r.pairs):
        ref = oracle_mod.match(r.images[i], r.images[j])
        np.testing.assert_array_equal(outs[k].row_top2.cpu().numpy(), ref.row_top2)
        np.testing.assert_array_equal(outs[k].col_top2.cpu().numpy(), ref.col_top2)
        np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)


def test_batch_host_buffers_and_reuse(serac, oracle_mod):
    """match_batch on pinned host images (shared between pairs), outputs in pinned
    host memory, then a second call into the same outputs: both equal the oracle."""
    imgs_np = [S.make_pair(7, 70, k, 900 + 300 * k, 10, 0.0, 0.05).a for k in range(4)]
    for k in range(3):  # plant rows of image k into image k + 1
        imgs_np[k + 1][: 200] = imgs_np[k][100:300]
    imgs = [torch.from_numpy(x).pin_memory() for x in imgs_np]
    idx = [(0, 1), (1, 2), (2, 3), (0, 3), (3, 0)]
    pairs = [(imgs[i], imgs[j]) for i, j in idx]
    outs = serac.match_batch(pairs, host_out=True, top2=True)
    torch.cuda.synchronize()
    for rep in range(2):
        for k, (i, j) in enumerate(idx):
            ref = oracle_mod.match(imgs_np[i], imgs_np[j])
            assert not outs[k].count.is_cuda
            np.testing.assert_array_equal(outs[k].row_top2.numpy(), ref.row_top2)
            np.testing.assert_array_equal(outs[k].col_top2.numpy(), ref.col_top2)
            np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)
        for o in outs:
            o.count.fill_(-99)
            o.row_top2.fill_(-7)
        outs = serac.match_batch(pairs, outs=outs)
        torch.cuda.synchronize()


def test_batch_host_images_over_chunks(serac, oracle_mod):
    """188 pairs of 16 shared pinned host images: two launch chunks, the second
    chunk's new images staged on the side stream while the first computes, and its
    pairs also reusing images the first chunk staged."""
    imgs_np = [S.make_pair(8, 71, k, 300 + 97 * k, 10, 0.0, 0.05).a for k in range(16)]
    for k in range(15):  # plant rows of image k into image k + 1
        imgs_np[k + 1][: 150] = imgs_np[k][50:200]
    imgs = [torch.from_numpy(x).pin_memory() for x in imgs_np]
    idx = [(i, j) for i in range(12) for j in range(12) if i != j][:128]   # chunk 0: images 0..11
    idx += [(i, j) for i in range(12, 16) for j in range(16) if i != j][:72]  # chunk 1 adds 12..15
    pairs = [(imgs[i], imgs[j]) for i, j in idx]
    outs = serac.match_batch(pairs, top2=True)
    torch.cuda.synchronize()
    for k, (i, j) in enumerate(idx):
        ref = oracle_mod.match(imgs_np[i], imgs_np[j])
        np.testing.assert_array_equal(outs[k].row_top2.cpu().numpy(), ref.row_top2)
        np.testing.assert_array_equal(outs[k].col_top2.cpu().numpy(), ref.col_top2)
        np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)


def test_batch_concurrent_host_threads(serac, oracle_mod):
    """Two host threads run multi-chunk batches at the same time, each on its own
    stream and workspace (each thread stages its later chunks on its own side stream);
    a third batch runs on the legacy default stream.  Every output equals the oracle."""
    import threading
    imgs_np = [S.make_pair(9, 72, k, 200 + 61 * k, 10, 0.0, 0.05).a for k in range(13)]
    for k in range(12):
        imgs_np[k + 1][: 100] = imgs_np[k][20:120]
    refs = {}
    # 156 pairs in two chunks; image 12 is first used by the second chunk
    order = sorted(((i, j) for i in range(13) for j in range(13) if i != j), key=lambda t: (max(t), t))

    def batch(kind):
        imgs = [torch.from_numpy(x).pin_memory() if kind == "host" else _dev(x) for x in imgs_np]
        return order, [(imgs[i], imgs[j]) for i, j in order]

    results, errors = {}, []

    def worker(name, kind):
        try:
            idx, pairs = batch(kind)
            st = torch.cuda.Stream()
            ws = serac.workspace(serac.batch_workspace_size(pairs), torch.device("cuda", 0))
            outs = None
            for _ in range(3):
                outs = serac.match_batch(pairs, workspace_t=ws, stream=st, outs=outs)
            st.synchronize()
            results[name] = (idx, outs)
        except Exception as exc:  # reported by the main thread
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(n, k)) for n, k in (("t0", "host"), ("t1", "device"))]
    for t in threads:
        t.start()
    idx, pairs = batch("device")
    legacy = serac.match_batch(pairs, stream=torch.cuda.default_stream())
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    results["legacy"] = (idx, legacy)
    for name, (idx, outs) in results.items():
        for k, (i, j) in enumerate(idx):
            if (i, j) not in refs:
                refs[(i, j)] = oracle_mod.match(imgs_np[i], imgs_np[j]).matches
            np.testing.assert_array_equal(outs[k].result().numpy(), refs[(i, j)], err_msg=f"{name} pair {k}")


def test_exact_beside_a_saturating_stream(serac, oracle_mod):
    """Calls that run while another stream keeps the SMs busy (a chain of large bf16
    GEMMs) still return exact results: the match kernel's blocks only wait on blocks
    that already run (tickets), whatever else occupies the GPU."""
    p = S.single_pair_2000(0)
    ref = oracle_mod.match(p.a, p.b)
    a, b = _dev(p.a), _dev(p.b)
    x = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(40):
            x = torch.nn.functional.normalize(x @ x, dim=1).to(torch.bfloat16)
    outs = [serac.match_pair(a, b, top2=True) for _ in range(25)]
    torch.cuda.synchronize()
    for o in outs:
        np.testing.assert_array_equal(o.result().numpy(), ref.matches)
        np.testing.assert_array_equal(o.row_top2.cpu().numpy(), ref.row_top2)
        np.testing.assert_array_equal(o.col_top2.cpu().numpy(), ref.col_top2)


def test_batch_ragged_256(serac, oracle_mod):
    """256 ragged pairs (1,000..16,384 features per image) through one match_batch:
    every pair compared in full with the oracle -- row top-2, column top-2 and the
    match list with its order."""
    sizes = S.ragged_sizes(0)
    pairs = [S.ragged_pair(0, k, sizes) for k in range(256)]
    dev = [(_dev(p.a), _dev(p.b)) for p in pairs]
    outs = serac.match_batch(dev, top2=True)
    torch.cuda.synchronize()
    for k, p in enumerate(pairs):
        ref = oracle_mod.match(p.a, p.b)
        o = outs[k]
        np.testing.assert_array_equal(o.row_top2.cpu().numpy(), ref.row_top2, err_msg=f"pair {k} rows")
        np.testing.assert_array_equal(o.col_top2.cpu().numpy(), ref.col_top2, err_msg=f"pair {k} columns")
        np.testing.assert_array_equal(o.result().numpy(), ref.matches, err_msg=f"pair {k} matches")


@pytest.mark.parametrize("ratio,angle", [(0.7, 0.6), (0.9, 0.8), (0.75, 0.5), (1.0, 0.9)])
def test_other_ratios_and_angles(serac, oracle_mod, ratio, angle):
    """Parameters other than 0.8 / 0.7 rad, derived by serac_default_params (and by the
    oracle separately), on the 2,000 x 2,000 pair and on a pair of ties."""
    p = serac.default_params(ratio, angle)
    q = oracle_mod.default_params(ratio, angle)
    assert (p.ratio_num_sq, p.ratio_den_sq, p.min_score) == (q.ratio_num_sq, q.ratio_den_sq, q.min_score)
    pr = S.single_pair_2000(0)
    out, ref = _assert_pair(serac, oracle_mod, pr.a, pr.b, p)
    assert len(ref.matches) > 0
    rng = np.random.default_rng(12)
    vals = np.array([0, 1, 2, 255], np.uint8)
    a = vals[rng.integers(0, 4, size=(400, 128))]
    b = vals[rng.integers(0, 4, size=(300, 128))]
    a[rng.random(a.shape) < 0.6] = 0
    b[rng.random(b.shape) < 0.6] = 0
    b[100:140] = b[1]
    p.norm_sq = 3_000_000
    _assert_pair(serac, oracle_mod, a, b, p)


@pytest.mark.parametrize("cap", [1, 700, 1999, 2000, 5000])
def test_feature_cap(serac, oracle_mod, cap):
    """max_features = K matches only the first K descriptors of each image (the match
    cap of the SERAC page, section 'Memory'): equal to the oracle under the same cap and
    to a plain match of the truncated images."""
    pr = S.make_pair(3, 67, 0, 2000, 3000, 0.3, 0.05)
    p = serac.default_params(max_features=cap)
    out, ref = _assert_pair(serac, oracle_mod, pr.a, pr.b, p)
    k_a, k_b = min(cap, 2000), min(cap, 3000)
    assert out.row_top2.shape[0] == max(k_a, 1) and out.col_top2.shape[0] == max(k_b, 1)
    plain = oracle_mod.match(pr.a[:k_a], pr.b[:k_b])
    np.testing.assert_array_equal(out.result().numpy(), plain.matches)
    # the same cap through match_batch, next to an uncapped-size pair
    outs = serac.match_batch([(_dev(pr.a), _dev(pr.b)), (_dev(pr.b[:900]), _dev(pr.a[:500]))], p, top2=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(outs[0].result().numpy(), ref.matches)
    ref2 = oracle_mod.match(pr.b[:900], pr.a[:500], oracle_mod.Params(max_features=cap))
    np.testing.assert_array_equal(outs[1].result().numpy(), ref2.matches)
    np.testing.assert_array_equal(outs[1].row_top2.cpu().numpy()[:min(cap, 900)], ref2.row_top2)


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_batch_equals_unsharded(serac, oracle_mod, world):
    """A batch split over `world` GPUs by shard_pairs, each shard run by its own
    match_batch (here one after another on one GPU), gives every pair exactly the
    match list (and top-2 tables) of the unsharded match_batch."""
    sizes = S.ragged_sizes(0)[:40] // 4
    pairs_np = [S.make_pair(9, 68, k, int(sizes[k, 0]), int(sizes[k, 1]), 0.15, 0.05) for k in range(40)]
    dev = [(_dev(p.a), _dev(p.b)) for p in pairs_np]
    whole = serac.match_batch(dev, top2=True)
    torch.cuda.synchronize()
    seen = []
    for rank in range(world):
        mine, outs = serac.match_batch_shard(dev, rank, world, top2=True)
        torch.cuda.synchronize()
        seen += mine
        for k, o in zip(mine, outs):
            assert torch.equal(o.result(), whole[k].result()), (rank, k)
            assert torch.equal(o.row_top2, whole[k].row_top2) and torch.equal(o.col_top2, whole[k].col_top2)
    assert sorted(seen) == list(range(40))
    for k in (0, 17, 39):
        np.testing.assert_array_equal(whole[k].result().numpy(), oracle_mod.match(pairs_np[k].a, pairs_np[k].b).matches)


def test_batch_survey_spot_50(serac, oracle_mod):
    """100 images x 8,192 (4,950 pairs) through match_batch; the 50 seeded pairs
    are checked in full against the oracle, every pair for order and range."""
    r = S.survey_100x8192(0)
    imgs = [_dev(x) for x in r.images]
    outs = serac.match_batch([(imgs[i], imgs[j]) for i, j in r.pairs])
    torch.cuda.synchronize()
    counts = torch.cat([o.count for o in outs]).cpu().numpy()
    assert counts.min() >= 0 and counts.max() <= 8192
    for k in S.survey_spot_pairs(0).tolist():
        i, j = r.pairs[k]
        ref = oracle_mod.match(r.images[i], r.images[j])
        np.testing.assert_array_equal(outs[k].result().numpy(), ref.matches)
    # planted neighbours match, far pairs (ring distance > 3) almost never do
    near = [k for k, (i, j) in enumerate(r.pairs) if min((j - i) % 100, (i - j) % 100) <= 3]
    assert counts[near].min() > 500
