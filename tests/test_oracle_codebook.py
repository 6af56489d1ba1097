"""Pins of the oracle's rotation and codebook builder against scipy routines, closed forms and
the invariants of Lloyd's algorithm."""
import numpy as np
import pytest
from scipy import special, stats

import synth
from oracle import codebook as ocb
from oracle import workloads as ow


def test_haar_rotation_is_orthogonal():
    for d in (8, 64, 128):
        Pi = ocb.haar_rotation(synth.rotation_gaussian(9, d))
        assert np.abs(Pi.T @ Pi - np.eye(d)).max() < 1e-12
        assert abs(abs(np.linalg.det(Pi)) - 1.0) < 1e-10
        P32 = Pi.astype(np.float32).astype(np.float64)
        assert np.abs(P32.T @ P32 - np.eye(d)).max() < 2e-6


def test_haar_rotation_law():
    # Under the Haar law every entry is a coordinate of a uniform unit vector: the diagonal is
    # sign-symmetric and Pi_ii^2 ~ Beta(1/2, (d-1)/2). Plain QR without the sign fix fails this
    # (LAPACK's Householder QR gives a diagonal of fixed sign).
    d = 16
    diag = np.array([np.diag(ocb.haar_rotation(np.random.default_rng([5, s]).standard_normal((d, d))))
                     for s in range(2000)])
    for i in (0, d // 2, d - 1):
        frac = np.mean(diag[:, i] > 0)
        assert abs(frac - 0.5) < 0.05
        assert stats.kstest(diag[:, i] ** 2, stats.beta(0.5, (d - 1) / 2).cdf).pvalue > 1e-3


def test_k2_radii_closed_form_matches_beta_quantile():
    for d, N in [(64, 16), (64, 256), (128, 64)]:
        a, b = ocb.companding_beta_params(d, 2)
        want = np.sqrt(special.betaincinv(a, b, (np.arange(N) + 0.5) / N))
        np.testing.assert_allclose(ocb.companded_radii(d, 2, N), want, rtol=1e-12, atol=1e-15)
    r = ocb.companded_radii(64, 2, 16)
    np.testing.assert_allclose(r[[0, 7, 15]], [0.04452, 0.19688, 0.44131], atol=5e-6)


def test_radii_follow_companded_density_counts():
    # Points with radius below rho: their fraction matches the Beta(k/2, a+1) law of rho^2
    # (Bennett-Gersho point density ~ f^(k/(k+2))), checked by numerical integration.
    d, k, N = 64, 4, 1024
    r = ocb.companded_radii(d, k, N)
    assert np.all(np.diff(r) > 0) and r[-1] < 1
    a = k * (d - k - 2) / (2 * (k + 2))
    for rho in (0.1, 0.2, 0.3):
        s = np.linspace(0, rho ** 2, 20001)
        dens = s ** (k / 2 - 1) * (1 - s) ** a
        full = np.linspace(0, 1, 200001)
        frac = np.trapezoid(dens, s) / np.trapezoid(full ** (k / 2 - 1) * (1 - full) ** a, full)
        assert abs(np.mean(r < rho) - frac) < 1.5 / N


def test_spiral_uses_golden_angle():
    C = ocb.spiral_codebook(64, 32)
    ang = np.unwrap(np.arctan2(C[:, 1], C[:, 0]))
    step = np.mod(np.diff(np.arctan2(C[:, 1], C[:, 0])), 2 * np.pi)
    np.testing.assert_allclose(step, np.pi * (3 - np.sqrt(5)), atol=1e-12)
    np.testing.assert_allclose(np.hypot(C[:, 0], C[:, 1]), ocb.companded_radii(64, 2, 32), rtol=1e-13)
    assert ang.size == 32


def test_roberts_constants_are_polynomial_roots():
    assert abs(ocb.roberts_root(1) - (1 + np.sqrt(5)) / 2) < 1e-14
    for k in (2, 4, 8, 64):
        phi = ocb.roberts_root(k)
        roots = np.roots([1] + [0] * (k - 1) + [-1, -1])
        real = max(r.real for r in roots if abs(r.imag) < 1e-9)
        assert abs(phi - real) < 1e-9


def test_kronecker_directions_unit_and_quasi_uniform():
    U = ocb.kronecker_directions(4096, 4, 0.5)
    np.testing.assert_allclose(np.linalg.norm(U, axis=1), 1.0, rtol=1e-13)
    # Uniform on S^3: each coordinate squared ~ Beta(1/2, 3/2); the mean direction is near 0.
    assert stats.kstest(U[:, 0] ** 2, stats.beta(0.5, 1.5).cdf).pvalue > 1e-3
    assert np.linalg.norm(U.mean(axis=0)) < 0.02


def test_source_points_law():
    g = synth.source_gaussians(1, 20000, 64)
    Y = ocb.source_points(g, 2)
    t = np.sum(Y ** 2, axis=1)
    assert stats.kstest(t, stats.beta(1, 31).cdf).pvalue > 1e-3


def _train(k, T=30000, d=64, seed=1):
    return ocb.source_points(np.random.default_rng(seed).standard_normal((T, d)), k)


def test_lloyd_mse_non_increasing_and_falls_with_N():
    Y = _train(2)
    last = np.inf
    for N in (4, 16, 64, 256):
        C, hist = ocb.lloyd(ocb.spiral_codebook(64, N), Y, 15)
        assert all(b <= a * (1 + 1e-12) for a, b in zip(hist, hist[1:]))
        assert hist[-1] < last
        last = hist[-1]


def test_vector_beats_scalar_at_matched_rate():
    # Section 3.2 / 4.1: at b = 2 bits per coordinate the k = 2, N = 16 code has lower MSE per
    # coordinate than the scalar (k = 1, N = 4) Lloyd-Max quantiser on the same source.
    Y = _train(2, T=60000)
    C2, h2 = ocb.lloyd(ocb.spiral_codebook(64, 16), Y, 30)
    y1 = Y[:, :1]
    C1, h1 = ocb.lloyd(np.quantile(y1, [0.125, 0.375, 0.625, 0.875])[:, None], y1, 60)
    assert h2[-1] / 2 < h1[-1]


def test_workload_codebooks_shapes_and_restart_choice():
    for cfg in (1, 2):
        w = synth.WORKLOADS[cfg]
        C = ow.codebook(cfg)
        assert C.shape == (w.N, w.k) and C.dtype == np.float32 and np.all(np.isfinite(C))
        assert np.unique(C, axis=0).shape[0] == w.N
    Pi = ow.rotation(2)
    assert Pi.dtype == np.float32 and Pi.shape == (64, 64)


def test_fibonacci_sphere_equal_area_and_golden_azimuth():
    # k = 3 directions (section 2.2, Fibonacci sphere). Heights are the centres of N equal slabs,
    # so by Archimedes' hat-box theorem every cap z > z0 holds its area's share of points to within
    # one point; consecutive azimuths differ by the golden angle; spacing is ~3.09 / sqrt(N).
    for N in (16, 64, 512, 2048):
        u = ocb.fibonacci_sphere(N)
        np.testing.assert_allclose(np.linalg.norm(u, axis=1), 1.0, atol=1e-14)
        np.testing.assert_allclose(np.sort(u[:, 2]), -1.0 + (2.0 * np.arange(N) + 1.0) / N, atol=1e-14)
        for z0 in np.linspace(-0.95, 0.95, 13):
            assert abs(np.sum(u[:, 2] > z0) - N * (1.0 - z0) / 2.0) <= 1.0
        az = np.arctan2(u[:, 1], u[:, 0])
        step = np.mod(np.diff(az), 2 * np.pi)
        np.testing.assert_allclose(step, np.pi * (3.0 - np.sqrt(5.0)), atol=1e-9)
        D = np.linalg.norm(u[:, None] - u[None], axis=2)
        np.fill_diagonal(D, 9.0)
        assert D.min() * np.sqrt(N) > 3.0


def test_fibsphere_codebook_pairs_radii_and_directions():
    d = 96
    for N in (8, 64, 512):
        C = ocb.initial_codebook("fibsphere", d, 3, N)
        r = np.linalg.norm(C, axis=1)
        np.testing.assert_allclose(r, ocb.companded_radii(d, 3, N), rtol=1e-13)
        u = C / r[:, None]
        S = ocb.fibonacci_sphere(N)
        # the directions are the Fibonacci sphere's, each used once
        match = np.argmin(np.linalg.norm(u[:, None] - S[None], axis=2), axis=1)
        assert np.array_equal(np.sort(match), np.arange(N))
        m = ocb.golden_stride(N)
        assert np.gcd(m, N) == 1 and abs(m - N / ocb.GOLDEN_RATIO) < 2
        if N >= 64:
            # the stride decorrelates radius from height (pairing in order would give about -1)
            assert abs(np.corrcoef(r, u[:, 2])[0, 1]) < 0.2
    with pytest.raises(ValueError):
        ocb.initial_codebook("fibsphere", 96, 2, 16)


def test_k3_vector_beats_scalar_at_matched_rate():
    # b = 2 bits per coordinate at d = 96: the k = 3, N = 64 Fibonacci-sphere code refined by Lloyd
    # has lower MSE per coordinate than the scalar (k = 1, N = 4) Lloyd-Max quantiser.
    g = np.random.default_rng(12).standard_normal((60000, 96))
    Y = ocb.source_points(g, 3)
    C3, h3 = ocb.lloyd(ocb.initial_codebook("fibsphere", 96, 3, 64), Y, 30)
    y1 = Y[:, :1]
    C1, h1 = ocb.lloyd(np.quantile(y1, [0.125, 0.375, 0.625, 0.875])[:, None], y1, 60)
    assert h3[-1] / 3 < h1[-1]
