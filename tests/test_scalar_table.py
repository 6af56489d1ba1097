"""The scalar Lloyd-Max table of the comparison codec (k = 1: normalise, rotate, quantise each
rotated coordinate with one scalar table [FibQuant §1]) against closed forms, numerical quadrature
and the oracle's Monte Carlo Lloyd iteration."""
import numpy as np
import pytest
from scipy import integrate, special

from oracle import codebook as ocb
from random_access_kv_gb300 import codebook as pcb


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_d3_marginal_is_uniform_so_the_table_is_the_uniform_quantiser(N):
    # One coordinate of a uniform point on the 2-sphere is uniform on [-1, 1] (Archimedes): the
    # Lloyd-Max quantiser of a uniform law has equal cells and midpoints, MSE (2/N)^2 / 12.
    C, mse = pcb.scalar_lloyd_max(3, N)
    np.testing.assert_allclose(C[:, 0], -1.0 + (2.0 * np.arange(N) + 1.0) / N, atol=1e-11)
    assert mse == pytest.approx((2.0 / N) ** 2 / 12.0, rel=1e-9)


@pytest.mark.parametrize("d", [16, 64, 128])
def test_one_bit_table_is_the_half_space_centroid(d):
    # N = 2: levels -+E[Y | Y > 0] = 2 * integral_0^1 y (1 - y^2)^m dy / B(1/2, m + 1).
    m = (d - 3) / 2
    c = 2.0 / (2.0 * (m + 1.0)) / special.beta(0.5, m + 1.0)
    C, mse = pcb.scalar_lloyd_max(d, 2)
    np.testing.assert_allclose(C[:, 0], [-c, c], rtol=1e-12)
    assert mse == pytest.approx(1.0 / d - c * c, rel=1e-9)


@pytest.mark.parametrize("d,N", [(64, 8), (128, 16)])
def test_centroid_and_midpoint_conditions_by_quadrature(d, N):
    m = (d - 3) / 2
    f = lambda y: (1.0 - y * y) ** m
    Z = integrate.quad(f, -1, 1, epsabs=0, epsrel=1e-13)[0]
    C, mse = pcb.scalar_lloyd_max(d, N)
    c = C[:, 0]
    assert np.all(np.diff(c) > 0) and np.allclose(c, -c[::-1], atol=1e-12)
    t = np.concatenate([[-1.0], 0.5 * (c[1:] + c[:-1]), [1.0]])
    err = 0.0
    for j in range(N):
        P = integrate.quad(f, t[j], t[j + 1], epsabs=0, epsrel=1e-12)[0] / Z
        M = integrate.quad(lambda y: y * f(y), t[j], t[j + 1], epsabs=0, epsrel=1e-12)[0] / Z
        assert M / P == pytest.approx(c[j], rel=1e-8, abs=1e-12)
        err += integrate.quad(lambda y: (y - c[j]) ** 2 * f(y), t[j], t[j + 1], epsabs=0, epsrel=1e-12)[0] / Z
    assert mse == pytest.approx(err, rel=1e-7)


def test_gaussian_limit_matches_max_table():
    # For large d, sqrt(d) y is close to N(0, 1): Max's (1960) Gaussian Lloyd-Max levels and MSEs.
    d = 1 << 14
    table = {4: ([0.4528, 1.5104], 0.1175), 8: ([0.2451, 0.7560, 1.3439, 2.1520], 0.03454)}
    for N, (levels, mse_g) in table.items():
        C, mse = pcb.scalar_lloyd_max(d, N)
        np.testing.assert_allclose(C[N // 2:, 0] * np.sqrt(d), levels, atol=2e-3)
        assert mse * d == pytest.approx(mse_g, rel=3e-3)


def test_oracle_monte_carlo_lloyd_agrees():
    # The oracle's generic Lloyd iteration on draws of the k = 1 block source, started from the
    # companded Kronecker initialisation, reaches the same table within sampling error.
    d, N = 64, 8
    r = np.random.default_rng(11)
    Y = ocb.source_points(r.standard_normal((400_000, d)), 1)
    C0 = ocb.initial_codebook("kronecker", d, 1, N)
    C_mc, hist = ocb.lloyd(C0, Y, iters=300, tol=1e-12)
    C, mse = pcb.scalar_lloyd_max(d, N)
    np.testing.assert_allclose(np.sort(C_mc[:, 0]) * np.sqrt(d), C[:, 0] * np.sqrt(d), atol=0.02)
    assert hist[-1] == pytest.approx(mse, rel=0.02)
