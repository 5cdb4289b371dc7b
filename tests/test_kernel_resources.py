"""Resource checks of the kernels at compile time (nvcc only, no GPU): the fused
kernel must keep its 576 threads within one SM's register file without spilling, and
the staging and match kernels must stay at 32 registers per thread, the size that
lets their four-warp blocks run beside a fused CTA (an SM sub-partition holding five
fused warps of 96 registers has room for one more warp of 32)."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "top_ratio_test_gb300", "csrc")


def _ptxas_report(src: str) -> dict:
    from top_ratio_test_gb300 import _build
    nvcc = _build._nvcc()
    if shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        cmd = [nvcc, "-Xptxas=-v", *_build.NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o",
               os.path.join(tmp, "k.o")]
        r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out, cur = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            out[cur] = {}
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            out[cur]["spill"] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            out[cur]["regs"] = int(m.group(1))
    return out


def _entry(report: dict, name: str) -> list:
    return [v for k, v in report.items() if name in k]


def test_fused_kernel_fits_without_spills():
    rep = _ptxas_report("fused.cu")
    ks = _entry(rep, "fused_top2_kernel")
    assert ks, rep
    for k in ks:
        assert k.get("spill", 0) == 0, k
        assert k["regs"] * 576 <= 65536, k


def test_stage_and_match_kernels_fit_beside_a_fused_cta():
    rep = _ptxas_report("finish.cu")
    for name in ("stage_kernel", "match_kernel"):
        ks = _entry(rep, name)
        assert ks, (name, rep)
        for k in ks:
            assert k["regs"] <= 32, (name, k)
            assert k.get("spill", 0) == 0, (name, k)


def test_topk_merge_kernel_without_spills():
    rep = _ptxas_report("topk.cu")
    ks = _entry(rep, "topk_merge_kernel")
    assert len(ks) == 2, rep   # the K = 4 and K = 8 builds
    for k in ks:
        assert k.get("spill", 0) == 0, k
