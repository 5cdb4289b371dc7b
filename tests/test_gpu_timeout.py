"""Failure detection on the GPU without a fault: a bounded wait is made to run out
(the test hook stops the TMA producer from issuing copies, so the operands the MMA
waits for never arrive), and the call must report SERAC_ETIMEOUT through `count`
after the wait's limit, leaving the context usable for an exact next call."""
import time

import numpy as np
import pytest
import torch

import sift_synth as S

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout(oracle_mod):
    import top_ratio_test_gb300 as serac
    assert serac.device_check() == serac.OK
    p = S.make_pair(8, 80, 0, 700, 900, 0.3, 0.05)
    a = torch.from_numpy(p.a).cuda()
    b = torch.from_numpy(p.b).cuda()
    ref = oracle_mod.match(p.a, p.b)
    serac.inject_timeout(True)
    t0 = time.perf_counter()
    out = serac.match_pair(a, b, top2=True)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(out.count.item()) == serac.ETIMEOUT
    assert 1.5 < dt < 30.0  # the 2 s limit ran out; nothing waited without bound
    with pytest.raises(serac.SeracError) as e:
        out.result()
    assert e.value.status == serac.ETIMEOUT
    # the hook was consumed by that call: the next one runs normally and exactly
    out2 = serac.match_pair(a, b, top2=True)
    np.testing.assert_array_equal(out2.result().numpy(), ref.matches)
    np.testing.assert_array_equal(out2.row_top2.cpu().numpy(), ref.row_top2)
    np.testing.assert_array_equal(out2.col_top2.cpu().numpy(), ref.col_top2)
