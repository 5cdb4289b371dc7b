"""The C ABI from a plain C program (tests/c_abi_client.c): it compiles against
include/serac.h and links libserac_gb300.so here; on a GPU its results equal the
oracle's."""
import os
import subprocess

import numpy as np
import pytest

import sift_synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    from top_ratio_test_gb300 import _build
    _build.build()
    exe = str(tmp_path / "c_abi_client")
    lib_dir = os.path.join(ROOT, "top_ratio_test_gb300")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c_abi_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lserac_gb300", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = _compile(tmp_path)
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_client_matches_oracle(tmp_path, oracle_mod):
    exe = _compile(tmp_path)
    p = S.make_pair(9, 90, 0, 1500, 2100, 0.3, 0.05)
    fa, fb, fo = tmp_path / "a.u8", tmp_path / "b.u8", tmp_path / "out.bin"
    p.a.tofile(fa)
    p.b.tofile(fb)
    r = subprocess.run([exe, str(fa), str(p.a.shape[0]), str(fb), str(p.b.shape[0]), str(fo)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    raw = np.fromfile(fo, dtype=np.int32)
    n = int(raw[0])
    na, nb = p.a.shape[0], p.b.shape[0]
    matches = raw[1:1 + 2 * n].reshape(n, 2)
    o = 1 + 2 * n
    row_top2 = raw[o:o + 4 * na].reshape(na, 4)
    o += 4 * na
    col_top2 = raw[o:o + 4 * nb].reshape(nb, 4)
    o += 4 * nb
    top3_s = raw[o:o + 3 * na].reshape(na, 3)
    top3_i = raw[o + 3 * na:].reshape(na, 3)
    ref = oracle_mod.match(p.a, p.b)
    np.testing.assert_array_equal(matches, ref.matches)
    np.testing.assert_array_equal(row_top2, ref.row_top2)
    np.testing.assert_array_equal(col_top2, ref.col_top2)
    rs, ri = oracle_mod.row_topk(p.a, p.b, 3)
    np.testing.assert_array_equal(top3_s, rs)
    np.testing.assert_array_equal(top3_i, ri)
