"""The C ABI without a GPU: the library builds, loads and exports every function the header
declares; host-side argument checks answer before any device work."""
import ctypes

import numpy as np
import pytest

from random_access_kv_gb300 import _binding as fb
from random_access_kv_gb300 import build as fbuild


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fb.lib()


def test_exports_every_header_symbol(L):
    names = fb.header_symbols()
    assert "fq_encode" in names and "fq_decode_gather" in names and "fq_codebook_load" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fb._SIGNATURES)


def test_strerror_and_null_context(L):
    assert fb.strerror(0) == "ok"
    assert "invalid" in fb.strerror(1)
    assert L.fq_code_words(None, 10) == -1
    assert L.fq_record_bits(None) == -1
    assert L.fq_encode(None, None, 5, None, None, 0, None) == fb.FQ_EINVAL
    assert L.fq_decode_gather(None, None, None, 5, None, 5, None, None) == fb.FQ_EINVAL
    assert L.fq_shape(None, None, None, None) == fb.FQ_EINVAL
    assert L.fq_attend(None, None, None, 10, None, 1, 1, 5, 0, 5, 5, 0.1, None, None) == fb.FQ_EINVAL
    assert L.fq_centroid_sums(None, None, 10, None, None, None, None, None) == fb.FQ_EINVAL
    assert L.fq_selftest_wait(None, 1000, None) == fb.FQ_EINVAL
    assert L.fq_encode_append(None, None, 1, 1, 4, 0, None, None, None) == fb.FQ_EINVAL
    assert L.fq_decode(None, None, None, 4, None, None) == fb.FQ_EINVAL
    L.fq_destroy(None)


def _load(L, C, Pi):
    h = ctypes.c_void_p()
    C = np.ascontiguousarray(C, dtype=np.float32)
    Pi = np.ascontiguousarray(Pi, dtype=np.float32)
    rc = L.fq_codebook_load(ctypes.byref(h), C.ctypes.data, C.shape[0], C.shape[1], Pi.ctypes.data,
                            Pi.shape[0], 0)
    return rc, h.value


@pytest.mark.parametrize("N,k,d", [(12, 2, 64), (1, 2, 64), (256, 3, 64), (256, 2, 80), (256, 3, 128), (131072, 2, 64),
                                   (65536, 2, 64), (16, 64, 64), (256, 128, 128)])
def test_codebook_load_rejects_unsupported_shapes(L, N, k, d):
    rc, h = _load(L, np.zeros((N, k)), np.eye(d))
    assert rc == fb.FQ_EINVAL and not h


def test_codebook_load_rejects_non_finite(L):
    C = np.zeros((16, 2))
    C[3, 1] = np.nan
    assert _load(L, C, np.eye(64))[0] == fb.FQ_EINVAL
    P = np.eye(64)
    P[0, 5] = np.inf
    assert _load(L, np.zeros((16, 2)), P)[0] == fb.FQ_EINVAL


def test_codebook_load_without_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _load(L, np.zeros((16, 2)), np.eye(64))
    assert rc == fb.FQ_ENODEV and not h


def test_archive_null_context_and_host_checks(L):
    assert L.fa_segments(None, 10) == -1
    assert L.fa_params(None, None, None, None) == fb.FQ_EINVAL
    assert L.fa_vertex_table(None, None) == fb.FQ_EINVAL
    assert L.fa_encode(None, None, 1, 4, 8, 0, None, None) == fb.FQ_EINVAL
    assert L.fa_decode(None, None, 1, 8, 8, None, None) == fb.FQ_EINVAL
    assert L.fa_access(None, None, 1, 8, 8, None, 1, None, None) == fb.FQ_EINVAL
    assert L.fa_status(None, None, None) == fb.FQ_EINVAL
    L.fa_destroy(None)
    h = ctypes.c_void_p()
    # parameter checks answer before any device is touched
    assert L.fa_create(ctypes.byref(h), 1, 0.1, 4, 0) == fb.FQ_EINVAL and not h.value
    assert L.fa_create(ctypes.byref(h), 8192, 1e-4, 2, 0) == fb.FQ_EINVAL
    assert L.fa_create(ctypes.byref(h), 16, 0.2, 4, 0) == fb.FQ_EINVAL        # r above the limit
    assert L.fa_create(ctypes.byref(h), 16, float("nan"), 4, 0) == fb.FQ_EINVAL
    r = 0.75 * L.fa_ratio_limit(16)
    assert L.fa_create(ctypes.byref(h), 16, r, L.fa_max_segment(16, r) + 1, 0) == fb.FQ_EINVAL
    assert L.fa_create(ctypes.byref(h), 16, r, 0, 0) == fb.FQ_EINVAL
    assert L.fa_create(None, 16, r, 4, 0) == fb.FQ_EINVAL


def test_archive_limits_match_the_oracle(L):
    # The disjointness limit and the segment-length bound are host arithmetic, stated in the library
    # and (separately) in the oracle; both must give the same lengths.
    from oracle import fractal as ofa
    for N in (2, 3, 4, 5, 16, 64, 100, 256, 1000, 4096):
        assert L.fa_ratio_limit(N) == pytest.approx(ofa.ratio_limit(N), rel=1e-15)
        for rho in (0.1, 0.25, 0.5, 0.6, 0.75, 0.9, 0.99, 1.0, 1.2):
            r = rho * ofa.ratio_limit(N)
            assert L.fa_max_segment(N, r) == ofa.max_segment(N, r), (N, rho)
    assert L.fa_ratio_limit(1) == 0.0 and L.fa_max_segment(1, 0.1) == 0 and L.fa_max_segment(8, -0.1) == 0


def test_codebook_load_accepts_k3_at_d96(L):
    # d = 96 with k = 3 (the Fibonacci-sphere codebook) passes the shape checks; without a GPU
    # the load then stops at the device check. k = 3 with d = 64 or 128 does not divide d.
    rc, h = _load(L, np.zeros((64, 3)), np.eye(96))
    assert rc in (fb.FQ_ENODEV, fb.FQ_OK) and (rc != fb.FQ_OK or h)
    if h:
        L.fq_destroy(ctypes.c_void_p(h))
    for d in (64, 128):
        rc, h = _load(L, np.zeros((64, 3)), np.eye(d))
        assert rc == fb.FQ_EINVAL and not h
    rc, h = _load(L, np.zeros((64, 5)), np.eye(96))
    assert rc == fb.FQ_EINVAL


def test_archive_segment_bound_agrees_with_the_oracle_everywhere(L):
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    from oracle import fractal as ofa

    @hyp.settings(max_examples=300, deadline=None, derandomize=True)
    @hyp.given(st.integers(2, 4096), st.floats(0.0, 1.1))
    def check(N, rho):
        r = rho * ofa.ratio_limit(N)
        assert L.fa_max_segment(N, r) == ofa.max_segment(N, r)

    check()
