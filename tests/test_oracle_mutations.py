"""Plants plausible mistakes in the oracle (on the CPU, through monkeypatching) and checks that at
least one pin catches each: a pinned oracle must not survive a dropped term, a wrong sign or index,
or a transposed operand."""
import numpy as np
import pytest

from oracle import codebook as ocb
from oracle import fibquant as fq

import test_oracle_codebook as tc
import test_oracle_encode as te


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_transposed_rotation_is_caught(monkeypatch):
    orig = fq.rotate_normalise
    monkeypatch.setattr(fq, "rotate_normalise", lambda x, Pi, nu: orig(x, np.asarray(Pi).T, nu))
    assert _fails(te.test_decode_encode_round_trip_on_codeword_vectors, 64, 4, 256)


def test_transposed_inverse_rotation_is_caught(monkeypatch):
    def bad(nu, idx, C, Pi):
        M, nb = idx.shape
        y = np.asarray(C)[idx].reshape(M, -1)
        return np.asarray(nu)[:, None] * (y @ np.asarray(Pi).T)
    monkeypatch.setattr(fq, "decode", bad)
    assert _fails(te.test_decode_encode_round_trip_on_codeword_vectors, 64, 2, 16)


def test_dropped_norm_is_caught(monkeypatch):
    monkeypatch.setattr(fq, "row_norms", lambda x: np.ones(np.asarray(x).shape[0]))
    assert _fails(te.test_norm_against_library_and_closed_form)
    assert _fails(te.test_decode_encode_round_trip_on_codeword_vectors, 64, 4, 256)


def test_expanded_form_without_norm_term_is_caught(monkeypatch):
    def bad(P, C, chunk_elems=0):
        return np.argmin(-2.0 * np.asarray(P) @ np.asarray(C).T, axis=1)
    monkeypatch.setattr(fq, "nearest_codeword", bad)
    assert _fails(te.test_nearest_codeword_matches_kdtree)


def test_wrong_tie_break_is_caught(monkeypatch):
    def bad(P, C, chunk_elems=0):
        d2 = np.sum((np.asarray(P)[:, None, :] - np.asarray(C)[None]) ** 2, axis=2)
        return d2.shape[1] - 1 - np.argmin(d2[:, ::-1], axis=1)
    monkeypatch.setattr(fq, "nearest_codeword", bad)
    assert _fails(te.test_codewords_map_to_themselves_and_ties_go_low)


def test_msb_first_packing_is_caught(monkeypatch):
    orig = fq.pack
    def bad(idx, B):
        idx = np.asarray(idx)
        rev = np.zeros_like(idx)
        for t in range(B):
            rev |= ((idx >> t) & 1) << (B - 1 - t)
        return orig(rev, B)
    monkeypatch.setattr(fq, "pack", bad)
    for B, idx, want in te._golden_pack_vectors():
        if _fails(te.test_pack_golden, B, idx, want):
            return
    pytest.fail("MSB-first packing survived the golden vectors")


def test_missing_sign_fix_is_caught(monkeypatch):
    monkeypatch.setattr(ocb, "haar_rotation", lambda G: np.linalg.qr(np.asarray(G))[0])
    assert _fails(tc.test_haar_rotation_law)


def test_shifted_radius_quantile_is_caught(monkeypatch):
    def bad(d, k, N):
        p = (np.arange(N) + 1.0) / (N + 1)
        return np.sqrt(1.0 - (1.0 - p) ** (4.0 / d))
    monkeypatch.setattr(ocb, "companded_radii", bad)
    assert _fails(tc.test_k2_radii_closed_form_matches_beta_quantile)


def test_wrong_source_law_is_caught(monkeypatch):
    monkeypatch.setattr(ocb, "source_points", lambda g, k: np.asarray(g)[:, :k] / np.sqrt(np.asarray(g).shape[1]))
    assert _fails(tc.test_source_points_law)


# Iterated-map archive ("Fractal KV-Cache Archives", Method 1)

import test_oracle_fractal as tf
from oracle import fractal as ofa


def test_swapped_contraction_weights_are_caught(monkeypatch):
    # p_k = p_{k-1} + r (V - p_{k-1}) puts weight r on the vertex instead of 1 - r
    def bad(symbols, N, r, start=(0.0, 0.0), V=None):
        V = ofa.vertices(N) if V is None else V
        x, y = start
        for c in symbols:
            x, y = x + r * (V[c, 0] - x), y + r * (V[c, 1] - y)
        return float(x), float(y)
    monkeypatch.setattr(ofa, "encode_segment", bad)
    assert _fails(tf.test_encode_matches_unrolled_recurrence_to_40_digits, 16, 0.75, 9)


def test_clockwise_polygon_is_caught(monkeypatch):
    orig = ofa.vertices
    monkeypatch.setattr(ofa, "vertices", lambda N: orig(N) * np.array([1.0, -1.0]))
    assert _fails(tf.test_vertices_regular_polygon)
    assert _fails(tf.test_encode_matches_unrolled_recurrence_to_40_digits, 16, 0.75, 9)


def test_start_at_a_vertex_is_caught(monkeypatch):
    orig = ofa.encode_segment
    monkeypatch.setattr(ofa, "encode_segment",
                        lambda s, N, r, start=(0.0, 0.0), V=None: orig(s, N, r, start=(1.0, 0.0), V=V))
    assert _fails(tf.test_encode_matches_unrolled_recurrence_to_40_digits, 3, 0.5, 12)


def test_inverse_without_vertex_term_is_caught(monkeypatch):
    def bad(anchor, length, N, r, stop=0, V=None):
        x, y = anchor
        out = []
        for _ in range(length - 1, stop - 1, -1):
            c = ofa.nearest_cell(x, y, N, r)
            out.append(c)
            x, y = x / r, y / r
        return out[::-1]
    monkeypatch.setattr(ofa, "decode_segment", bad)
    assert _fails(tf.test_round_trip_every_string, 3, 9)


def test_optimistic_segment_bound_is_caught(monkeypatch):
    # a bound that ignores the amplification allows segments too long to decode
    orig = ofa.max_segment
    monkeypatch.setattr(ofa, "max_segment", lambda N, r, cap=64: 3 * orig(N, r, cap))
    assert _fails(tf.test_round_trip_at_the_segment_limit, 256)


def test_in_order_radius_pairing_is_caught(monkeypatch):
    # pairing the n-th radius with the n-th (height-ordered) sphere point ties radius to height
    from oracle import codebook as ocb2
    import test_oracle_codebook as tcb
    monkeypatch.setattr(ocb2, "golden_stride", lambda N: 1)
    assert _fails(tcb.test_fibsphere_codebook_pairs_radii_and_directions)
