"""Pins of the oracle's encoder, decoder and bit layout against things other than itself:
library routines, closed forms, hand-worked bit vectors and invariants."""
import os

import numpy as np
import pytest
from scipy import spatial, stats

import synth
from oracle import codebook as ocb
from oracle import fibquant as fq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_rate_formula():
    # b = log2(N)/k bits per coordinate; R = d b bits per vector.
    assert fq.record_bits(64, 2, 256) == 256 and 256 / 64 == 4.0
    assert fq.record_bits(64, 4, 1024) == 160 and 160 / 64 == 2.5
    assert fq.record_bits(128, 8, 4096) == 192 and 192 / 128 == 1.5
    assert fq.record_bits(64, 64, 4096) == 12 and 12 / 64 == 0.1875
    with pytest.raises(ValueError):
        fq.bits_per_index(12)
    with pytest.raises(ValueError):
        fq.record_bits(64, 3, 16)


def test_norm_against_library_and_closed_form():
    x = np.array([[3.0, 4.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0]])
    np.testing.assert_array_equal(fq.row_norms(x), [5.0, 0.0, 2.0])
    r = np.random.default_rng(0).standard_normal((257, 64)).astype(np.float16)
    np.testing.assert_allclose(fq.row_norms(r), np.linalg.norm(r.astype(np.float64), axis=1), rtol=1e-14)


def test_rotation_gives_unit_vectors_and_identity_case():
    Pi = ocb.haar_rotation(synth.rotation_gaussian(1, 64))
    x = synth.kv_tensor(1).astype(np.float64)[:500]
    nu = fq.row_norms(x)
    u = fq.rotate_normalise(x, Pi, nu)
    np.testing.assert_allclose(np.linalg.norm(u, axis=1), 1.0, atol=1e-12)
    # With the identity rotation u is x / ||x||, written out by hand for one vector.
    u1 = fq.rotate_normalise(np.array([[3.0, 0.0, 4.0, 0.0]]), np.eye(4), np.array([5.0]))
    np.testing.assert_array_equal(u1, [[0.6, 0.0, 0.8, 0.0]])
    # A zero row stays zero.
    assert not np.any(fq.rotate_normalise(np.zeros((1, 4)), np.eye(4), np.zeros(1)))


def test_theorem1_block_norms_are_beta_isotropic():
    # Theorem 1 / section 2.1: after norm + Haar rotation a k-block has ||u_b||^2 ~ Beta(k/2, (d-k)/2).
    Pi = ocb.haar_rotation(synth.rotation_gaussian(1, 64))
    x = synth.kv_tensor(1).astype(np.float64)
    u = fq.rotate_normalise(x, Pi, fq.row_norms(x))
    for k in (2, 8):
        t = np.sum(u[:, :k] ** 2, axis=1)
        assert stats.kstest(t, stats.beta(k / 2, (64 - k) / 2).cdf).pvalue > 1e-3
        assert abs(t.mean() - k / 64) < 4 * np.sqrt(stats.beta(k / 2, (64 - k) / 2).var() / t.size)


def test_theorem1_over_rotation_draws_anisotropic_input():
    # One fixed, strongly anisotropic vector; the law comes from the Haar draw of the rotation.
    d, k = 64, 4
    x = np.ones((1, d))
    x[0, 5] = 400.0
    x[0, :10] *= 7.0
    t = []
    for s in range(2000):
        Pi = ocb.haar_rotation(np.random.default_rng([77, s]).standard_normal((d, d)))
        u = fq.rotate_normalise(x, Pi, fq.row_norms(x))
        t.append(np.sum(u[0, 8:8 + k] ** 2))
    assert stats.kstest(t, stats.beta(k / 2, (d - k) / 2).cdf).pvalue > 1e-3


def test_nearest_codeword_matches_kdtree():
    r = np.random.default_rng(3)
    for k, N in [(2, 16), (2, 256), (4, 64), (8, 128), (64, 32)]:
        C = r.standard_normal((N, k)) * 0.3
        P = r.standard_normal((700, k)) * 0.3
        _, ref = spatial.cKDTree(C).query(P)
        np.testing.assert_array_equal(fq.nearest_codeword(P, C), ref)


def test_nearest_codeword_scalar_midpoint_rule():
    # k = 1: the textbook rule of a scalar quantiser, decision thresholds at midpoints.
    r = np.random.default_rng(4)
    levels = np.sort(r.standard_normal(9))
    C = levels[r.permutation(9)][:, None]
    p = r.standard_normal(3000)
    order = np.argsort(C[:, 0])
    mids = 0.5 * (C[order[1:], 0] + C[order[:-1], 0])
    ref = order[np.searchsorted(mids, p)]
    np.testing.assert_array_equal(fq.nearest_codeword(p[:, None], C), ref)


def test_codewords_map_to_themselves_and_ties_go_low():
    C = np.asarray(ocb.spiral_codebook(64, 256))
    np.testing.assert_array_equal(fq.nearest_codeword(C, C), np.arange(256))
    D = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0], [0.0, 1.0]])
    np.testing.assert_array_equal(fq.nearest_codeword(D, D), [0, 1, 0, 1])
    # A point equidistant from two codewords takes the lower index.
    np.testing.assert_array_equal(fq.nearest_codeword(np.array([[0.5, 0.5]]), D[::-1]), [0])


def _golden_pack_vectors():
    rows = []
    with open(os.path.join(GOLDEN, "pack_vectors.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            B, idx, hexbytes = line.split()
            rows.append((int(B), [int(v) for v in idx.split(",")], bytes.fromhex(hexbytes)))
    return rows


@pytest.mark.parametrize("B,idx,want", _golden_pack_vectors())
def test_pack_golden(B, idx, want):
    words = fq.pack(np.array(idx)[None, :], B)
    got = words.astype("<u4").tobytes()
    assert got[:len(want)] == want
    assert not any(got[len(want):])
    np.testing.assert_array_equal(fq.unpack(words, 1, len(idx), B)[0], idx)
    np.testing.assert_array_equal(fq.record_indices(words, 0, len(idx), B), idx)


@pytest.mark.parametrize("nb,B", [(32, 4), (32, 8), (16, 10), (16, 12), (1, 12), (3, 5)])
def test_pack_round_trip_and_fixed_address(nb, B):
    r = np.random.default_rng(nb * 100 + B)
    M = 77
    idx = r.integers(0, 1 << B, size=(M, nb))
    w = fq.pack(idx, B)
    assert w.size == (M * nb * B + 31) // 32
    np.testing.assert_array_equal(fq.unpack(w, M, nb, B), idx)
    for m in (0, 1, 38, M - 1):
        np.testing.assert_array_equal(fq.record_indices(w, m, nb, B), idx[m])
    # A record written alone lands at bit m*R of the stream: packing rows m.. gives the same
    # bits shifted by m*R.
    R = nb * B
    tail = fq.pack(idx[5:], B)
    bits_all = np.unpackbits(w.view(np.uint8), bitorder="little")
    bits_tail = np.unpackbits(tail.view(np.uint8), bitorder="little")
    np.testing.assert_array_equal(bits_all[5 * R:M * R], bits_tail[:(M - 5) * R])


def _equal_norm_codebook(k, d, N, seed):
    r = np.random.default_rng(seed)
    C = r.standard_normal((N, k))
    return C / np.linalg.norm(C, axis=1, keepdims=True) * np.sqrt(k / d)


@pytest.mark.parametrize("d,k,N", [(64, 2, 16), (64, 4, 256), (128, 8, 64), (64, 64, 128)])
def test_decode_encode_round_trip_on_codeword_vectors(d, k, N):
    # If every codeword has norm sqrt(k/d), any concatenation y has norm 1, and x = nu Pi^T y is
    # encoded to exactly those indices and decoded back to x (section 2.3 decoder, closed form).
    C = _equal_norm_codebook(k, d, N, d + k + N)
    Pi = ocb.haar_rotation(np.random.default_rng(d * k).standard_normal((d, d)))
    r = np.random.default_rng(5)
    M = 50
    idx = r.integers(0, N, size=(M, d // k))
    nu = r.uniform(0.1, 30.0, size=M)
    x = nu[:, None] * (C[idx].reshape(M, d) @ Pi)
    nu2, idx2 = fq.encode(x, C, Pi)
    np.testing.assert_allclose(nu2, nu, rtol=1e-13)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_allclose(fq.decode(nu2, idx2, C, Pi), x, rtol=0, atol=1e-12 * nu.max())


def test_decode_identity_rotation_by_hand():
    C = np.array([[0.6, 0.8], [0.0, 0.0], [1.0, 0.0], [0.0, -1.0]])
    nu = np.array([5.0, 2.0])
    idx = np.array([[0, 1], [3, 2]])
    want = np.array([[3.0, 4.0, 0.0, 0.0], [0.0, -2.0, 2.0, 0.0]])
    np.testing.assert_array_equal(fq.decode(nu, idx, C, np.eye(4)), want)
    # and the encoder maps these vectors back (norm 5 and 2*sqrt(2))
    nu2, idx2 = fq.encode(want, C, np.eye(4))
    np.testing.assert_allclose(nu2, [5.0, 2.0 * np.sqrt(2.0)])
    np.testing.assert_array_equal(idx2[0], [0, 1])


def test_zero_row_encodes_to_zero():
    C = np.asarray(ocb.spiral_codebook(8, 16))
    nu, idx = fq.encode(np.zeros((2, 8)), C, np.eye(8))
    assert not nu.any() and not idx.any()
    assert not fq.decode(nu, idx, C, np.eye(8)).any()
