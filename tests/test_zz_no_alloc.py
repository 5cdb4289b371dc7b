"""match_pair_noalloc: matching on the library's built-in scratch, for callers that may
not allocate device memory (host applications that own every allocation, real-time
loops, fixed-footprint tools).  Its results must equal match_pair's on the same inputs,
on two calls in a row (the scratch keeps the previous call's contents, so the second
call checks that nothing stale leaks through).  This file is named to be collected
last, so a run that stops at the first failure has run every other test first."""
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


def _outputs(o):
    torch.cuda.synchronize()
    return o.result().numpy(), o.row_top2.cpu().numpy(), o.col_top2.cpu().numpy()


def test_noalloc_matches_match_pair_twice(serac):
    first = S.single_pair_2000(0)
    second = S.make_pair(4, 63, 0, 1500, 2600, 0.3, 0.05)
    for p in (first, second):
        a = torch.from_numpy(p.a).cuda()
        b = torch.from_numpy(p.b).cuda()
        ref = _outputs(serac.match_pair(a, b, top2=True))
        got = _outputs(serac.match_pair_noalloc(a, b, top2=True))
        for x, y in zip(got, ref):
            np.testing.assert_array_equal(x, y)
        assert len(ref[0]) > 0


def test_noalloc_rejects_oversized_pairs(serac):
    n = 32768
    assert serac.pair_workspace_size(16384, 16384) <= serac.NOALLOC_SCRATCH_BYTES
    assert serac.pair_workspace_size(n, n) > serac.NOALLOC_SCRATCH_BYTES
    a = torch.zeros((n, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(serac.SeracError) as e:
        serac.match_pair_noalloc(a, a)
    assert e.value.status == serac.EWORKSPACE
