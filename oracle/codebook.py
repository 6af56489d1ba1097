"""fp64 oracle of the FibQuant codebook and shared rotation (TEST INFRASTRUCTURE ONLY).

Restates [FibQuant §2.1] (the spherical-Beta source) and [FibQuant §2.2] (radii by
Bennett-Gersho companding, quasi-uniform directions, multi-restart Lloyd refinement) in plain
numpy/scipy. Random draws come in as arguments (from ``synth``).

Readings of the page where it is open:
  * rotation: Pi = Q diag(sign(diag R)) for the QR factorisation G = Q R of a d x d standard
    Gaussian; the sign fix makes the law of Pi exactly Haar. u = Pi x.
  * radii: Gersho's optimal point density lambda ~ f^(k/(k+2)) for the block density
    f(y) ~ (1 - |y|^2)^((d-k-2)/2) on the unit k-ball. In t = rho^2 the point count is then
    Beta(k/2, a+1), a = k (d-k-2) / (2 (k+2)); r_n = sqrt(BetaQuantile((n + 1/2) / N)).
    For k = 2 this is the closed form r_n = sqrt(1 - (1 - (n+1/2)/N)^(4/d)).
  * k = 2 directions: planar Fibonacci spiral, angle n * 2 pi (1 - 1/phi), paired with r_n.
  * k = 3 directions: the Fibonacci sphere, point j at height z_j = 1 - (2j + 1)/N and azimuth j times
    the golden angle. Its points are ordered by height, so radius n (also ordered) takes point
    j = (n m) mod N, m the odd integer nearest N / phi coprime to N (a golden-ratio stride), which
    spreads consecutive radii over the sphere as the k = 2 spiral's golden angle spreads them
    over the circle.
  * k >= 4 directions: Roberts-Kronecker points t_n = frac(s + (n+1) alpha), alpha_j = phi_k^-j
    (j = 1..k, phi_k the real root > 1 of x^(k+1) = x + 1; the sequence starts at its first
    term, so that codeword 0 is not the centre point t = s), mapped to the sphere by the inverse
    normal CDF and normalisation; codeword n = r_n u_n. For k = d the codewords are the unit
    directions themselves (the source is then the unit sphere).
  * Lloyd: training points y = g_{1..k} / ||g|| for g ~ N(0, I_d) (exact draws from f_{d,k});
    nearest-codeword assignment, then each codeword moves to the mean of its cell (an empty cell
    keeps its codeword; no renormalisation). Restart r >= 1 starts from the initialisation
    rotated by a seeded k x k Haar matrix; the lowest final MSE wins, ties to the lowest r.
"""
from __future__ import annotations

import numpy as np
from scipy import special


def haar_rotation(G) -> np.ndarray:
    """Pi = Q diag(sign(diag R)) with G = Q R [FibQuant §1 and §2.1: shared Haar rotation]."""
    Q, R = np.linalg.qr(np.asarray(G, dtype=np.float64))
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s[None, :]


def source_points(g, k: int) -> np.ndarray:
    """Draws of the spherical-Beta source f_{d,k}: the first k coordinates of g / ||g|| for rows
    g ~ N(0, I_d), i.e. one k-block of a Haar-uniform unit vector [FibQuant §2.1]."""
    g = np.asarray(g, dtype=np.float64)
    return g[:, :k] / np.sqrt(np.sum(g * g, axis=1))[:, None]


def companding_beta_params(d: int, k: int) -> tuple[float, float]:
    """Parameters (k/2, a+1) of the Beta law of t = rho^2 under the companded point density."""
    a = k * (d - k - 2) / (2.0 * (k + 2))
    return k / 2.0, a + 1.0


def companded_radii(d: int, k: int, N: int) -> np.ndarray:
    """r_n = sqrt(Beta quantile at (n + 1/2)/N) [FibQuant §2.2, radii by Bennett-Gersho
    companding]. k = 2 uses the closed form; k >= 3 uses scipy's inverse regularised beta."""
    p = (np.arange(N) + 0.5) / N
    if k == 2:
        return np.sqrt(1.0 - (1.0 - p) ** (4.0 / d))
    a, b = companding_beta_params(d, k)
    return np.sqrt(special.betaincinv(a, b, p))


GOLDEN_RATIO = (1.0 + 5.0 ** 0.5) / 2.0


def spiral_codebook(d: int, N: int) -> np.ndarray:
    """k = 2 planar Fibonacci spiral with companded radii [FibQuant §2.2, 'Golden Quantizer']."""
    r = companded_radii(d, 2, N)
    theta = np.arange(N) * (2.0 * np.pi * (1.0 - 1.0 / GOLDEN_RATIO))
    return np.stack([r * np.cos(theta), r * np.sin(theta)], axis=1)


def fibonacci_sphere(N: int) -> np.ndarray:
    """k = 3 directions [FibQuant §2.2, 'Fibonacci sphere']: point j at height z_j = 1 - (2j+1)/N,
    the centres of N slabs of equal height and hence (Archimedes' hat-box theorem) equal area, and
    azimuth j times the golden angle 2 pi (1 - 1/phi)."""
    j = np.arange(N, dtype=np.float64)
    z = 1.0 - (2.0 * j + 1.0) / N
    theta = j * (2.0 * np.pi * (1.0 - 1.0 / GOLDEN_RATIO))
    rho = np.sqrt(1.0 - z * z)
    return np.stack([rho * np.cos(theta), rho * np.sin(theta), z], axis=1)


def golden_stride(N: int) -> int:
    """The integer nearest N / phi that is coprime to N (the nearer below on a tie)."""
    target = N / GOLDEN_RATIO
    best = None
    for m in range(1, N + 1):
        if np.gcd(m, N) == 1 and (best is None or abs(m - target) < abs(best - target)):
            best = m
    return best


def fibsphere_codebook(d: int, N: int) -> np.ndarray:
    """k = 3 radial-angular initialisation: codeword n = r_n u_{(n m) mod N} with the companded
    radii r_n and the Fibonacci sphere u [FibQuant §2.2]."""
    r = companded_radii(d, 3, N)
    u = fibonacci_sphere(N)
    return r[:, None] * u[(np.arange(N) * golden_stride(N)) % N]


def roberts_root(k: int) -> float:
    """phi_k: the real root > 1 of x^(k+1) = x + 1, by bisection on [1, 2]."""
    lo, hi = 1.0, 2.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid ** (k + 1) - mid - 1.0 > 0:
            hi = mid
        else:
            lo = mid
    return 0.5 * (lo + hi)


def kronecker_directions(N: int, k: int, s: float) -> np.ndarray:
    """Unit directions from the k-dimensional Roberts-Kronecker sequence [FibQuant §2.2]."""
    phi = roberts_root(k)
    alpha = phi ** -np.arange(1, k + 1)
    t = np.mod(s + np.arange(1, N + 1)[:, None] * alpha[None, :], 1.0)
    if np.any(t <= 0.0) or np.any(t >= 1.0):
        raise ValueError("Kronecker point on the cube boundary")
    z = special.ndtri(t)
    return z / np.sqrt(np.sum(z * z, axis=1))[:, None]


def initial_codebook(kind: str, d: int, k: int, N: int, s: float = 0.5) -> np.ndarray:
    """Deterministic radial-angular initialisation [FibQuant §2.2]."""
    if kind == "spiral":
        if k != 2:
            raise ValueError("spiral codebook is k = 2")
        return spiral_codebook(d, N)
    if kind == "fibsphere":
        if k != 3:
            raise ValueError("Fibonacci-sphere codebook is k = 3")
        return fibsphere_codebook(d, N)
    u = kronecker_directions(N, k, s)
    if kind == "sphere":
        if k != d:
            raise ValueError("sphere codebook is k = d")
        return u
    if kind == "kronecker":
        return companded_radii(d, k, N)[:, None] * u
    raise ValueError(kind)


def assign(Y, C) -> np.ndarray:
    """Lloyd assignment: nearest codeword of every training point, ranked by the expanded
    distance ||c||^2 - 2 y.c (one BLAS product per chunk). This is codebook construction, not the
    encoder; the encoder's difference-form search is ``fibquant.nearest_codeword``."""
    Y = np.asarray(Y, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    cc = np.sum(C * C, axis=1)
    out = np.empty(Y.shape[0], dtype=np.int64)
    step = max(1, (1 << 24) // C.shape[0])
    for s in range(0, Y.shape[0], step):
        out[s:s + step] = np.argmin(cc[None, :] - 2.0 * (Y[s:s + step] @ C.T), axis=1)
    return out


def distortion(Y, C, idx) -> float:
    """Mean over training points of ||y - c_idx||^2."""
    e = np.asarray(Y, dtype=np.float64) - np.asarray(C, dtype=np.float64)[idx]
    return float(np.mean(np.sum(e * e, axis=1)))


def lloyd(C0, Y, iters: int, tol: float = 1e-6) -> tuple[np.ndarray, list]:
    """Lloyd iterations from C0 on training points Y [FibQuant §2.2, refinement]. Returns the
    refined codebook and the MSE of each codebook visited (first entry: C0)."""
    C = np.array(C0, dtype=np.float64, copy=True)
    Y = np.asarray(Y, dtype=np.float64)
    N, k = C.shape
    idx = assign(Y, C)
    hist = [distortion(Y, C, idx)]
    for _ in range(iters):
        counts = np.bincount(idx, minlength=N)
        sums = np.stack([np.bincount(idx, weights=Y[:, j], minlength=N) for j in range(k)], axis=1)
        filled = counts > 0
        C[filled] = sums[filled] / counts[filled, None]
        idx = assign(Y, C)
        hist.append(distortion(Y, C, idx))
        if hist[-2] - hist[-1] <= tol * hist[-2]:
            break
    return C, hist


def build_codebook(kind: str, d: int, k: int, N: int, Y, iters: int, restart_gaussians=(),
                   s: float = 0.5) -> tuple[np.ndarray, float]:
    """Multi-restart Lloyd refinement of the deterministic initialisation [FibQuant §2.2].
    ``restart_gaussians`` holds one k x k Gaussian per extra restart. Returns (C, MSE)."""
    C0 = initial_codebook(kind, d, k, N, s)
    starts = [C0] + [C0 @ haar_rotation(G).T for G in restart_gaussians]
    best, best_mse = None, np.inf
    for init in starts:
        C, hist = lloyd(init, Y, iters)
        if hist[-1] < best_mse:
            best, best_mse = C, hist[-1]
    return best, best_mse
