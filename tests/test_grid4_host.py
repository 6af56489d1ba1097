"""The k = 4 candidate grid's host builder (random_access_kv_gb300/csrc/fq_grid4.h), checked on the
CPU: for every probe point the cell the device's fp32 lattice arithmetic selects must list the
exact (double-precision brute force) nearest codeword, or the point must fall outside the grid,
where the device scans the whole codebook. Probes include points within 1e-4 of midpoints between
codewords, the hardest case for the lists' box tests. The lists must be ascending."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import workloads as ow

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("grid4") / "grid4_check")
    subprocess.run([cxx, "-O2", "-std=c++17", "-pthread", os.path.join(HERE, "grid4_check.cpp"), "-o", exe],
                   check=True)
    return exe


def run(checker, tmp_path, C, d, n_points, seed, drop=False):
    path = tmp_path / "C.f32"
    np.ascontiguousarray(C, dtype=np.float32).tofile(path)
    args = [checker, str(path), str(C.shape[0]), str(d), str(n_points), str(seed)] + (["1"] if drop else [])
    out = subprocess.run(args, check=True, capture_output=True, text=True).stdout.split()
    vals = dict(zip(out[0::2], out[1::2]))
    return int(vals["checked"]), int(vals["misses"]), int(vals["outside"])


def gaussian_codebook(N, d, seed):
    return np.random.default_rng(seed).standard_normal((N, 4)) / np.sqrt(d)


@pytest.mark.parametrize("N,d", [(16, 64), (256, 128), (4096, 64), (2, 64)])
def test_every_probe_finds_its_nearest_codeword_listed(checker, tmp_path, N, d):
    checked, misses, outside = run(checker, tmp_path, gaussian_codebook(N, d, N + d), d, 60000, 7)
    assert checked > 0.5 * 60000 and misses == 0


def test_workload_codebook(checker, tmp_path):
    checked, misses, outside = run(checker, tmp_path, ow.codebook(3), 64, 200000, 11)
    assert checked > 0.8 * 200000 and misses == 0


def test_duplicate_codewords_keep_the_lower_index_listed(checker, tmp_path):
    # Two codewords at the same point tie everywhere: neither is strictly dominated, so both stay
    # listed and the nearest by the lowest-index rule is found.
    C = gaussian_codebook(64, 64, 5)
    C[10] = C[3]
    checked, misses, outside = run(checker, tmp_path, C, 64, 60000, 3)
    assert misses == 0


def test_a_planted_list_error_is_caught(checker, tmp_path):
    # The check ignoring each list's first entry (as a builder that dropped it would) must fail.
    checked, misses, outside = run(checker, tmp_path, gaussian_codebook(256, 64, 9), 64, 20000, 5, drop=True)
    assert misses > 0.05 * checked
