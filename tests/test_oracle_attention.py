"""Pins of the attention oracle: scipy's softmax, invariants and closed forms."""
import numpy as np
from scipy import special

from oracle import attention as oat
from oracle import fibquant as ofq


def test_softmax_attention_matches_scipy():
    r = np.random.default_rng(0)
    q, K, V = r.standard_normal(16), r.standard_normal((40, 16)), r.standard_normal((40, 16))
    want = special.softmax(0.25 * (K @ q)) @ V
    np.testing.assert_allclose(oat.softmax_attention(q, K, V, 0.25), want, rtol=1e-13, atol=1e-14)


def test_softmax_attention_closed_forms():
    r = np.random.default_rng(1)
    V = r.standard_normal((7, 8))
    # equal scores: the mean of the values; one token: that value; a dominant score: its value
    np.testing.assert_allclose(oat.softmax_attention(np.zeros(8), r.standard_normal((7, 8)), V, 1.0),
                               V.mean(axis=0), rtol=1e-13)
    np.testing.assert_allclose(oat.softmax_attention(r.standard_normal(8), V[:1], V[:1], 3.0), V[0], rtol=1e-14)
    K = np.zeros((7, 8))
    K[3, 0] = 1e3
    q = np.zeros(8)
    q[0] = 1.0
    np.testing.assert_allclose(oat.softmax_attention(q, K, V, 1.0), V[3], atol=1e-12)


def test_attention_is_permutation_invariant_over_tokens():
    r = np.random.default_rng(2)
    q, K, V = r.standard_normal(8), r.standard_normal((30, 8)), r.standard_normal((30, 8))
    perm = r.permutation(30)
    np.testing.assert_allclose(oat.softmax_attention(q, K[perm], V[perm], 0.5),
                               oat.softmax_attention(q, K, V, 0.5), rtol=1e-12)


def test_attention_decode_uses_the_codec_decoder():
    # Keys and values built from codewords are decoded exactly, so the compressed attention equals
    # attention over the original vectors (section 2.3 decoder; section 5 fused attention).
    # The decoder's output is fixed independently of ofq.decode here: an orthogonal Pi built from
    # a permutation and signs maps concat(c) to a signed permutation of it.
    d, k, N, T = 16, 4, 32, 20
    r = np.random.default_rng(3)
    C = r.standard_normal((N, k))
    perm = r.permutation(d)
    Pi = np.zeros((d, d))
    Pi[np.arange(d), perm] = r.choice([-1.0, 1.0], size=d)
    idx_k, idx_v = r.integers(0, N, size=(T, d // k)), r.integers(0, N, size=(T, d // k))
    nu_k, nu_v = r.uniform(0.5, 3.0, size=T), r.uniform(0.5, 3.0, size=T)
    q = r.standard_normal((3, d))
    got = oat.attention_decode(q, nu_k, idx_k, nu_v, idx_v, C, Pi, 0.3)
    # x_hat = nu Pi^T y: component perm[i] of x_hat is sign_i * nu * y_i
    sign = Pi[np.arange(d), perm]
    def dec(nu, idx):
        y = C[idx].reshape(len(nu), d)
        x = np.zeros_like(y)
        x[:, perm] = sign * y * nu[:, None]
        return x
    K, V = dec(nu_k, idx_k), dec(nu_v, idx_v)
    for g in range(3):
        want = special.softmax(0.3 * (K @ q[g])) @ V
        np.testing.assert_allclose(got[g], want, rtol=1e-12, atol=1e-13)


def test_record_range_matches_single_record_reads():
    r = np.random.default_rng(4)
    for nb, B in [(32, 8), (16, 10), (16, 12), (1, 12), (8, 3)]:
        idx = r.integers(0, 1 << B, size=(70, nb))
        words = ofq.pack(idx, B)
        for m0, cnt in [(0, 70), (3, 17), (69, 1), (5, 0)]:
            got = ofq.record_range(words, m0, cnt, nb, B)
            np.testing.assert_array_equal(got, idx[m0:m0 + cnt].reshape(cnt, nb))
        np.testing.assert_array_equal(ofq.record_range(words, 11, 1, nb, B)[0],
                                      ofq.record_indices(words, 11, nb, B))


def test_cosine():
    a = np.array([[1.0, 0.0], [1.0, 1.0]])
    np.testing.assert_allclose(oat.cosine(a, np.array([[2.0, 0.0], [-1.0, -1.0]])), [1.0, -1.0])
