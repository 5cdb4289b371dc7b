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


def test_noalloc_allocates_nothing(serac):
    """After the first call in this context (which looks up the scratch's address),
    further calls through the raw C ABI change neither the device's free memory nor
    the caching allocator's reservations: no cudaMalloc, no cudaFree, nothing pooled."""
    import ctypes
    p = S.single_pair_2000(0)
    a = torch.from_numpy(p.a).cuda()
    b = torch.from_numpy(p.b).cuda()
    params = serac.default_params()
    o, c = serac._make_out(2000, 2000, a.device, None, True)
    ref = _outputs(serac.match_pair(a, b, top2=True))
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return serac.lib().match_pair_noalloc(a.data_ptr(), 2000, b.data_ptr(), 2000, ctypes.byref(params),
                                              ctypes.byref(c), stream)

    assert call() == serac.OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        assert call() == serac.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0
    for x, y in zip(_outputs(o), ref):
        np.testing.assert_array_equal(x, y)


def test_noalloc_rejects_oversized_pairs(serac):
    n = 32768
    assert serac.pair_workspace_size(16384, 16384) <= serac.NOALLOC_SCRATCH_BYTES
    assert serac.pair_workspace_size(n, n) > serac.NOALLOC_SCRATCH_BYTES
    a = torch.zeros((n, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(serac.SeracError) as e:
        serac.match_pair_noalloc(a, a)
    assert e.value.status == serac.EWORKSPACE
