"""C ABI checks that need no GPU: the library loads, exports every symbol the header
declares, and its host-only logic (parameters, workspace sizes, argument checks, the
work schedule) behaves as documented.  No call here reaches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def serac():
    from top_ratio_test_gb300 import _build
    _build.build()
    import top_ratio_test_gb300 as s
    return s


def _declared():
    src = open(os.path.join(ROOT, "include", "serac.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M))


def test_header_symbols_exported(serac):
    names = _declared()
    assert len(names) >= 10
    assert names == set(serac.EXPORTS)
    L = serac.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(serac):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert serac.status_str(s) != "unknown status"
    assert serac.status_str(7) == "unknown status"


def test_default_params(serac):
    p = serac.default_params(0.8, 0.7)
    assert (p.ratio_num_sq, p.ratio_den_sq, p.norm_sq, p.min_score, p.mutual, p.col_ratio) == \
        (16, 25, 262144, 200499, 1, 1)
    p = serac.default_params(0.75, 0.7)
    assert p.ratio_num_sq * 16 == p.ratio_den_sq * 9
    q = serac.Params()
    for bad in [(0.0, 0.7), (1.5, 0.7), (0.8, -0.1), (0.8, 2.0)]:
        assert serac.lib().serac_default_params(ctypes.byref(q), *bad) == serac.EINVAL
    assert serac.lib().serac_default_params(None, 0.8, 0.7) == serac.EINVAL


def test_workspace_sizes(serac):
    small = serac.pair_workspace_size(100, 100)
    big = serac.pair_workspace_size(8192, 8192)
    assert 0 < small < big
    # 2 images x 8192 rows x 256 B staged plus 16 B of keys per row and column
    assert abs(big - (2 * 8192 * 256 + 2 * 8192 * 16)) < 8192  # plus alignment padding
    assert serac.pair_workspace_size(0, 0) > 0


def test_bad_arguments_rejected_before_any_launch(serac):
    L = serac.lib()
    p = serac.default_params()
    cnt = ctypes.c_int32()
    out = serac._Out(16, 4, ctypes.addressof(cnt), None, None)
    ws = 1 << 20
    # null descriptors with n > 0
    assert L.match_pair(None, 4, 16, 4, ctypes.byref(p), ctypes.byref(out), 256, ws, None) == serac.EINVAL
    # negative size, size above the limit
    assert L.match_pair(16, -1, 16, 4, ctypes.byref(p), ctypes.byref(out), 256, ws, None) == serac.EINVAL
    assert L.match_pair(16, (1 << 24) + 1, 16, 4, ctypes.byref(p), ctypes.byref(out), 256, ws, None) == serac.EINVAL
    # misaligned descriptors
    assert L.match_pair(17, 4, 16, 4, ctypes.byref(p), ctypes.byref(out), 256, ws, None) == serac.EINVAL
    # no params / no outputs / no count
    assert L.match_pair(16, 4, 16, 4, None, ctypes.byref(out), 256, ws, None) == serac.EINVAL
    assert L.match_pair(16, 4, 16, 4, ctypes.byref(p), None, 256, ws, None) == serac.EINVAL
    out2 = serac._Out(16, 4, None, None, None)
    assert L.match_pair(16, 4, 16, 4, ctypes.byref(p), ctypes.byref(out2), 256, ws, None) == serac.EINVAL
    # misaligned optional top-2 output
    out3 = serac._Out(16, 4, ctypes.addressof(cnt), 20, None)
    assert L.match_pair(16, 4, 16, 4, ctypes.byref(p), ctypes.byref(out3), 256, ws, None) == serac.EINVAL
    # ratio denominator must be positive
    p0 = serac.default_params()
    p0.ratio_den_sq = 0
    assert L.match_pair(16, 4, 16, 4, ctypes.byref(p0), ctypes.byref(out), 256, ws, None) == serac.EINVAL
    # batch: negative count, null arrays
    assert L.match_batch(None, 2, ctypes.byref(p), None, 256, ws, None) == serac.EINVAL
    assert L.match_batch(None, -1, ctypes.byref(p), None, 256, ws, None) == serac.EINVAL


def test_noalloc_argument_checks(serac):
    """match_pair_noalloc rejects bad sizes before any CUDA call: out of range -> EINVAL,
    a workspace larger than the built-in scratch (after the feature cap) -> EWORKSPACE."""
    L = serac.lib()
    p = serac.default_params()
    cnt = ctypes.c_int32()
    out = serac._Out(16, 4, ctypes.addressof(cnt), None, None)
    assert L.match_pair_noalloc(16, -1, 16, 4, ctypes.byref(p), ctypes.byref(out), None) == serac.EINVAL
    assert L.match_pair_noalloc(16, (1 << 24) + 1, 16, 4, ctypes.byref(p), ctypes.byref(out), None) == serac.EINVAL
    assert L.match_pair_noalloc(16, 4, 16, 4, None, ctypes.byref(out), None) == serac.EINVAL
    big = 32768
    assert serac.pair_workspace_size(big, big) > serac.NOALLOC_SCRATCH_BYTES
    assert L.match_pair_noalloc(16, big, 32, big, ctypes.byref(p), ctypes.byref(out), None) == serac.EWORKSPACE
    p.max_features = -1
    assert L.match_pair_noalloc(16, 4, 16, 4, ctypes.byref(p), ctypes.byref(out), None) == serac.EINVAL


def test_feature_cap_params(serac):
    """max_features: 0 by default, negative rejected before any launch."""
    L = serac.lib()
    p = serac.default_params()
    assert p.max_features == 0
    assert serac.default_params(max_features=500).max_features == 500
    cnt = ctypes.c_int32()
    out = serac._Out(16, 4, ctypes.addressof(cnt), None, None)
    p.max_features = -3
    assert L.match_pair(16, 4, 16, 4, ctypes.byref(p), ctypes.byref(out), 256, 1 << 20, None) == serac.EINVAL
    assert L.match_batch(None, 0, ctypes.byref(p), None, 256, 1 << 20, None) == serac.EINVAL


def test_default_params_agree_with_the_oracle(serac, oracle_mod):
    """The library's integer parameters and the oracle's, derived separately from the
    same ratio and angle, agree (including non-default ratios and angles)."""
    for r, ang in [(0.8, 0.7), (0.7, 0.6), (0.9, 0.8), (0.75, 0.5), (1.0, 1.2), (0.6, 0.0)]:
        p = serac.default_params(r, ang)
        q = oracle_mod.default_params(r, ang)
        assert (p.ratio_num_sq, p.ratio_den_sq, p.norm_sq, p.min_score) == \
            (q.ratio_num_sq, q.ratio_den_sq, q.norm_sq, q.min_score), (r, ang)


def _tiles(na, nb):
    """Tiles of one row problem: 128-row tiles of the row side, 256-row tiles of the other."""
    return ((na + 127) // 128) * ((nb + 255) // 256) if na > 0 and nb > 0 else 0


def _pair_tiles(na, nb):
    """A pair is two row problems: A's rows against B, B's rows against A."""
    return _tiles(na, nb) + _tiles(nb, na)


def test_schedule_covers_every_tile_once(serac):
    # a single 8192 x 8192 pair on 152 CTAs: 2 x 2048 tiles dealt 26 or 27 per CTA
    chunks, pieces, npieces, cta = serac.schedule_describe([(8192, 8192)], 152)
    assert chunks == 1
    assert npieces == [152, 152] and pieces == 304
    assert sum(cta) == 2 * 64 * 32
    assert sorted(set(cta)) == [26, 27] and cta.count(27) == 4096 % 152


def test_schedule_small_pair_uses_every_cta(serac):
    # 2000 x 2000: two problems of 16 x 8 = 128 tiles; 152 CTAs take one or two tiles
    chunks, pieces, npieces, cta = serac.schedule_describe([(2000, 2000)], 152)
    assert npieces == [128, 128] and pieces == 256
    assert sum(cta) == 256 and sorted(set(cta)) == [1, 2]
    # a pair with fewer tiles than CTAs launches one CTA per tile
    chunks, pieces, npieces, cta = serac.schedule_describe([(300, 500)], 152)
    assert npieces == [_tiles(300, 500), _tiles(500, 300)] and sum(cta) == sum(npieces)
    assert cta[:sum(npieces)] == [1] * sum(npieces) and set(cta[sum(npieces):]) == {0}


def test_schedule_ragged_and_empty(serac):
    sizes = [(1000, 16384), (0, 500), (257, 0), (129, 255), (16384, 1000)]
    chunks, pieces, npieces, cta = serac.schedule_describe(sizes, 152)
    t = [x for na, nb in sizes for x in (_tiles(na, nb), _tiles(nb, na))]
    assert npieces == [min(152, x) for x in t]
    assert npieces[2:6] == [0, 0, 0, 0]
    assert pieces == sum(npieces)
    assert sum(cta) == sum(t)
    # tiles are dealt round-robin across problems: loads differ by at most one
    assert max(cta) - min(cta) <= 1


def test_schedule_balanced_over_many_pairs(serac):
    # 40 pairs of 1,700 + 1,700 tiles and 40 of 5 + 6 tiles: mixed sizes stay dealt one
    # piece per CTA, every CTA within one tile
    sizes = [(6400, 8704), (640, 256)] * 40
    chunks, pieces, npieces, cta = serac.schedule_describe(sizes, 152)
    assert chunks == 1
    t = [x for na, nb in sizes for x in (_tiles(na, nb), _tiles(nb, na))]
    assert npieces == [min(152, x) for x in t]
    assert sum(cta) == sum(t) and max(cta) - min(cta) <= 1


def test_schedule_small_pairs_in_whole_row_tiles(serac):
    # 128 pairs of 1024 x 1024 (8 row tiles x 4 column tiles per problem): dealt one
    # piece per row tile -- one segment each -- instead of one tile per CTA
    sizes = [(1024, 1024)] * 128
    chunks, pieces, npieces, cta = serac.schedule_describe(sizes, 152)
    assert npieces == [8] * 256 and pieces == 2048
    assert sum(cta) == 256 * 32 and max(cta) - min(cta) <= 4
    # the 66-pair ring of 8192 x 8192: whole rows of 32 tiles, 64 pieces per problem
    chunks, pieces, npieces, cta = serac.schedule_describe([(8192, 8192)] * 66, 152)
    assert npieces == [64] * 132 and sum(cta) == 132 * 2048 and max(cta) - min(cta) <= 32


def test_schedule_ragged_batch_stays_fine(serac):
    # pairs of mixed sizes: whole-row pieces would leave the CTAs several per cent
    # apart, so every problem is dealt one piece per CTA and the loads stay within one
    import sift_synth as S
    sizes = [(int(a), int(b)) for a, b in S.ragged_sizes(0)[:128]]
    chunks, pieces, npieces, cta = serac.schedule_describe(sizes, 152)
    t = [x for na, nb in sizes for x in (_tiles(na, nb), _tiles(nb, na))]
    assert npieces == [min(152, x) for x in t]
    assert sum(cta) == sum(t) and max(cta) - min(cta) <= 1


def test_schedule_large_batch_chunks(serac):
    sizes = [(8192, 8192)] * 300
    chunks, pieces, npieces, cta = serac.schedule_describe(sizes, 152)
    # at most 128 pairs per launch chunk (their tables travel as kernel parameters)
    assert chunks == 3
    assert npieces[:256] == [64] * 256 and pieces == 256 * 64
    assert sum(cta) == 128 * 2 * 2048 and max(cta) - min(cta) <= 32


def test_timeout_hook_is_host_only(serac):
    """The failure-detection hook only sets a host flag (the GPU test consumes it);
    clearing it leaves the next call untouched."""
    L = serac.lib()
    assert L.serac_test_inject_timeout(1) == 0
    assert L.serac_test_inject_timeout(0) == 0


def test_topk_argument_checks(serac):
    """serac_topk_pair rejects bad arguments before it touches a device; without a
    device the workspace query answers 0."""
    L = serac.lib()
    buf = ctypes.create_string_buffer(1 << 16)
    a = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256
    out = a + 4096
    assert L.serac_topk_pair(a, 10, a, 10, 0, out, out, None, a, 256, None) == serac.EINVAL   # k < 1
    assert L.serac_topk_pair(a, 10, a, 10, 9, out, out, None, a, 256, None) == serac.EINVAL   # k > 8
    assert L.serac_topk_pair(a, -1, a, 10, 2, out, out, None, a, 256, None) == serac.EINVAL   # n < 0
    assert L.serac_topk_pair(a, 10, a, 10, 2, None, out, None, a, 256, None) == serac.EINVAL  # no scores
    assert L.serac_topk_pair(a, 10, a, 10, 2, out, out + 2, None, a, 256, None) == serac.EINVAL  # misaligned
    assert L.serac_topk_pair(a + 8, 10, a, 10, 2, out, out, None, a, 256, None) == serac.EINVAL  # desc alignment
    assert L.serac_topk_pair(a, 10, a, 10, 2, out, out, out + 1, a, 256, None) == serac.EINVAL  # status alignment
    import torch
    if not torch.cuda.is_available():
        assert serac.topk_workspace_size(100, 100, 4) == 0
