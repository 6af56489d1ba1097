"""Pins of the iterated-map archive oracle ("Fractal KV-Cache Archives", Method 1).

What fixes each function independently of the oracle's own recurrence:
  * vertices: the regular polygon's closed forms and a 40-digit evaluation of cos and sin;
  * encode: the unrolled recurrence p_L = sum_j (1 - r) r^(L-j) V(c_j), evaluated to 40 digits;
  * ratio_limit: exact values at N = 2, 4, 6 and the touching of adjacent cells at the limit;
  * decode / access: exhaustive round trips of every string of a given length, adversarial strings
    at the segment-length limit, and failure a few symbols beyond it (the limit is not vacuous);
  * the page's suffix geometry: a shared suffix of length s contracts the distance by r^s.
"""
import itertools
import math

import mpmath
import numpy as np
import pytest

from oracle import fractal as fa


def test_vertices_regular_polygon():
    for N in (2, 3, 5, 256):
        V = fa.vertices(N)
        np.testing.assert_allclose(np.hypot(V[:, 0], V[:, 1]), 1.0, atol=4e-16)
        side = np.hypot(*(np.roll(V, -1, axis=0) - V).T)
        np.testing.assert_allclose(side, 2 * math.sin(math.pi / N), rtol=0, atol=2e-15)
        np.testing.assert_allclose(V.sum(axis=0), 0.0, atol=1e-13)
        assert V[0, 0] == 1.0 and V[0, 1] == 0.0
    mpmath.mp.dps = 40
    V = fa.vertices(7)
    for c in range(7):
        a = 2 * mpmath.pi * c / 7
        assert abs(V[c, 0] - float(mpmath.cos(a))) <= 2 ** -52
        assert abs(V[c, 1] - float(mpmath.sin(a))) <= 2 ** -52


def test_ratio_limit_closed_forms_and_touching_cells():
    assert fa.ratio_limit(2) == pytest.approx(0.5, abs=1e-16)
    assert fa.ratio_limit(4) == pytest.approx(math.sqrt(2) - 1, rel=1e-15)
    assert fa.ratio_limit(6) == pytest.approx(1 / 3, rel=1e-15)
    for N in (3, 8, 100):
        r = fa.ratio_limit(N)
        # adjacent cell centres (1 - r) V(c) are exactly 2 r apart at the limit: the discs touch
        assert 2 * (1 - r) * math.sin(math.pi / N) == pytest.approx(2 * r, rel=1e-14)
        assert fa.cell_margin(N, r) == pytest.approx(0.0, abs=1e-15)
        assert fa.cell_margin(N, 0.5 * r) > 0
        assert fa.max_segment(N, r) == 0 and fa.max_segment(N, 1.01 * r) == 0


@pytest.mark.parametrize("N,rho,L", [(2, 0.75, 20), (3, 0.5, 12), (16, 0.75, 9), (256, 0.75, 7)])
def test_encode_matches_unrolled_recurrence_to_40_digits(N, rho, L):
    mpmath.mp.dps = 40
    r = rho * fa.ratio_limit(N)
    rng = np.random.default_rng(N)
    for _ in range(5):
        sym = rng.integers(0, N, size=L)
        x, y = fa.encode_segment(sym, N, r)
        rm = mpmath.mpf(r)           # the method's r is the fp64 number
        ex = ey = mpmath.mpf(0)
        for j, c in enumerate(sym, start=1):
            a = 2 * mpmath.pi * int(c) / N
            w = (1 - rm) * rm ** (L - j)
            ex += w * mpmath.cos(a)
            ey += w * mpmath.sin(a)
        tol = 6 * fa.U / (1 - r)       # forward rounding plus the rounding of V, summed over steps
        assert abs(x - float(ex)) <= tol and abs(y - float(ey)) <= tol


def test_points_lie_in_their_cells():
    for N in (3, 64):
        r = 0.75 * fa.ratio_limit(N)
        V = fa.vertices(N)
        rng = np.random.default_rng(5)
        sym = rng.integers(0, N, size=40)
        x = y = 0.0
        for c in sym:
            x, y = fa.encode_segment([c], N, r, start=(x, y))
            d = np.hypot(x - (1 - r) * V[:, 0], y - (1 - r) * V[:, 1])
            assert d[c] <= r * (1 + 1e-12)
            assert np.all(np.delete(d, c) > r)
            assert fa.nearest_cell(x, y, N, r) == c


@pytest.mark.parametrize("N,L", [(2, 14), (3, 9), (5, 6)])
def test_round_trip_every_string(N, L):
    r = 0.75 * fa.ratio_limit(N)
    assert fa.max_segment(N, r) >= L
    V = fa.vertices(N)
    for sym in itertools.product(range(N), repeat=L):
        a = fa.encode_segment(sym, N, r, V=V)
        assert fa.decode_segment(a, L, N, r, V=V) == list(sym)


def adversarial(N: int, L: int, rng) -> np.ndarray:
    """Strings whose points sit at the far edge of their cells: runs of the vertex a quarter turn
    away from the next symbol, which puts the previous point near the unit circle, perpendicular
    to the next cell's direction."""
    out = []
    for _ in range(64):
        s = []
        while len(s) < L:
            c = int(rng.integers(N))
            side = (c + (N // 4 or 1) * (1 if rng.random() < 0.5 else -1)) % N
            s += [side] * int(rng.integers(1, 6)) + [c]
        out.append(s[:L])
    return np.array(out)


@pytest.mark.parametrize("N", [2, 3, 4, 16, 256, 1024, 4096])
def test_round_trip_at_the_segment_limit(N):
    r = 0.75 * fa.ratio_limit(N)
    L = fa.max_segment(N, r)
    assert L >= 4
    rng = np.random.default_rng(N + 1)
    V = fa.vertices(N)
    strings = np.concatenate([rng.integers(0, N, size=(200, L)), adversarial(N, L, rng)])
    for sym in strings:
        a = fa.encode_segment(sym, N, r, V=V)
        assert fa.decode_segment(a, L, N, r, V=V) == list(sym)


def test_decoding_fails_beyond_the_precision_limit():
    # Past the bound the amplified rounding error outgrows the cell margin: for N = 256 the error
    # after 9 backward steps is of order u (1/r)^9, far above the margin, so decoding breaks.
    N = 256
    r = 0.75 * fa.ratio_limit(N)
    L = fa.max_segment(N, r) + 3
    rng = np.random.default_rng(9)
    V = fa.vertices(N)
    bad = 0
    for sym in rng.integers(0, N, size=(20, L)):
        bad += fa.decode_segment(fa.encode_segment(sym, N, r, V=V), L, N, r, V=V) != list(sym)
    assert bad >= 10


def test_shared_suffix_contracts_by_r_to_the_s():
    # Points of strings that share their last s symbols differ by r^s times the difference of the
    # points before that suffix, hence by at most 2 r^s (both lie in the unit disc).
    N, L = 8, 12
    r = 0.5 * fa.ratio_limit(N)
    rng = np.random.default_rng(3)
    for s in (1, 3, 5):
        a, b = rng.integers(0, N, size=L), rng.integers(0, N, size=L)
        b[L - s:] = a[L - s:]
        pa, pb = np.array(fa.encode_segment(a, N, r)), np.array(fa.encode_segment(b, N, r))
        qa, qb = np.array(fa.encode_segment(a[:L - s], N, r)), np.array(fa.encode_segment(b[:L - s], N, r))
        assert np.linalg.norm(pa - pb) <= 2 * r ** s
        np.testing.assert_allclose(pa - pb, r ** s * (qa - qb), atol=16 * fa.U)


def test_streams_encode_decode_access_and_append():
    N, L, T_cap = 64, None, 50
    r = 0.75 * fa.ratio_limit(N)
    L = fa.max_segment(N, r)
    rng = np.random.default_rng(11)
    sym = rng.integers(0, N, size=(3, 37))
    A = fa.encode(sym, N, r, L, T_cap=T_cap)
    assert A.shape == (3, fa.segments(T_cap, L), 2)
    assert np.all(A[:, fa.segments(37, L):] == 0.0)
    np.testing.assert_array_equal(fa.decode(A, 37, N, r, L), sym)
    for q in range(3):
        for t in range(37):
            assert fa.access(A, 37, N, r, L, q, t) == sym[q, t]
    # appending in uneven chunks gives the same anchors bit for bit
    B = fa.encode(sym[:, :0], N, r, L, T_cap=T_cap)
    T = 0
    for n in (1, L - 1, 2, 2 * L + 3, 37 - (1 + L - 1 + 2 + 2 * L + 3)):
        B = fa.append(B, T, sym[:, T:T + n], N, r, L)
        T += n
    assert T == 37
    np.testing.assert_array_equal(B, A)


def test_symbol_range_is_checked():
    with pytest.raises(ValueError):
        fa.encode_segment([0, 4], 4, 0.1)
    with pytest.raises(IndexError):
        fa.access(np.zeros((1, 2, 2)), 5, 4, 0.1, 4, 0, 5)


def test_round_trip_property_over_alphabets_ratios_and_strings():
    """Any alphabet 2..4096, any ratio 10%..95% of the disjointness limit, any string of the
    longest allowed segment: the backward search returns the string."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(st.integers(2, 4096), st.floats(0.1, 0.95), st.integers(0, 2 ** 32 - 1))
    def check(N, rho, seed):
        r = rho * fa.ratio_limit(N)
        L = fa.max_segment(N, r)
        if L == 0:
            return
        sym = np.random.default_rng(seed).integers(0, N, size=L)
        assert fa.decode_segment(fa.encode_segment(sym, N, r), L, N, r) == list(sym)

    check()


def test_cell_margin_is_the_distance_from_a_cell_to_its_sector_edges():
    # Sample the boundary circle of cell c (radius r about (1 - r) V(c)) and measure each point's
    # distance to the two rays that bound the sector of c (angles 2 pi c / N +- pi / N); the
    # smallest distance is the margin g = (1 - r) sin(pi / N) - r.
    for N, rho in ((3, 0.5), (16, 0.75), (256, 0.9)):
        r = rho * fa.ratio_limit(N)
        c = 5 % N
        th = 2 * np.pi * c / N
        centre = (1 - r) * np.array([np.cos(th), np.sin(th)])
        phi = np.linspace(0, 2 * np.pi, 20001)
        pts = centre[None] + r * np.stack([np.cos(phi), np.sin(phi)], axis=1)
        dist = []
        for edge in (th - np.pi / N, th + np.pi / N):
            n = np.array([-np.sin(edge), np.cos(edge)])           # normal of the edge line
            dist.append(np.abs(pts @ n))
        got = np.min(np.minimum(*dist))
        assert got == pytest.approx(fa.cell_margin(N, r), rel=1e-6, abs=1e-12)
