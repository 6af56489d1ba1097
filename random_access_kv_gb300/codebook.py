"""Host-side builder of the shared FibQuant rotation and codebook (offline, numpy/scipy).

The codec's kernels take the codebook C [N, k] and rotation Pi [d, d] as inputs; this module makes
them from seeded random draws, following [FibQuant §2.1, §2.2] of the page "FibQuant: universal
vector quantisation for random-access KV-cache compression":

  rotation  Pi = Q diag(sign(diag R)) for G = Q R, G a d x d standard Gaussian (Haar law).
  radii     Bennett-Gersho companding of the spherical-Beta block law: the point density
            ~ f^(k/(k+2)) makes t = rho^2 of the codewords Beta(k/2, 1 + k(d-k-2)/(2(k+2)));
            r_n is the square root of that law's quantile at (n + 1/2)/N.
  angles    k = 2: Fibonacci spiral (golden angle per index). k = 3 ("fibsphere"): the Fibonacci
            sphere (heights at the centres of N equal slabs, golden-angle azimuths), visited with
            a golden-ratio stride m ~ N / phi coprime to N so that consecutive radii land far
            apart on the sphere. k >= 4: Roberts-Kronecker points
            frac(s + (n+1) phi_k^-j), j = 1..k, pushed through the inverse normal CDF and
            normalised; phi_k solves x^(k+1) = x + 1. k = d: the unit directions alone.
  Lloyd     multi-restart Lloyd on draws of the block source (first k coordinates of a Gaussian
            vector over its norm); restart r >= 1 rotates the start by a k x k Haar matrix; the
            lowest training MSE wins. ``build_gpu`` runs the same iterations through the library:
            the encoder assigns every block of every training row, ``fq_centroid_sums`` forms
            the centroids.

The scalar comparison codec of [FibQuant §1] (normalise, rotate, then quantise every rotated
coordinate with one scalar Lloyd-Max table) is the k = 1 case of the same interface; its table is
``scalar_lloyd_max``.

This is construction-time code, not part of the encode/decode path.
"""
from __future__ import annotations

import struct
import zlib

import numpy as np
from scipy import special


def haar(G: np.ndarray) -> np.ndarray:
    Q, R = np.linalg.qr(np.asarray(G, dtype=np.float64))
    d = np.diag(R)
    return Q * np.where(d < 0, -1.0, 1.0)


def radii(d: int, k: int, N: int) -> np.ndarray:
    alpha = 0.5 * k
    beta = 1.0 + k * (d - k - 2) / (2.0 * (k + 2))
    q = (np.arange(N, dtype=np.float64) + 0.5) / N
    return np.sqrt(special.betaincinv(alpha, beta, q))


def _roberts_phi(k: int) -> float:
    x = 2.0
    for _ in range(100):                    # Newton on x^(k+1) - x - 1, from above the root
        x -= (x ** (k + 1) - x - 1.0) / ((k + 1) * x ** k - 1.0)
    return x


def directions(N: int, k: int, s: float) -> np.ndarray:
    if k == 2:
        golden = np.pi * (3.0 - np.sqrt(5.0))
        a = golden * np.arange(N)
        return np.column_stack([np.cos(a), np.sin(a)])
    g = _roberts_phi(k)
    steps = np.power(g, -np.arange(1.0, k + 1.0))
    pts = np.modf(s + np.outer(np.arange(1, N + 1, dtype=np.float64), steps))[0]
    z = special.ndtri(pts)
    return z / np.linalg.norm(z, axis=1, keepdims=True)


def fibonacci_sphere(N: int) -> np.ndarray:
    z = np.linspace(1.0 - 1.0 / N, -1.0 + 1.0 / N, N)
    a = np.pi * (3.0 - np.sqrt(5.0)) * np.arange(N, dtype=np.float64)
    ring = np.sqrt(np.maximum(0.0, 1.0 - z * z))
    return np.column_stack([ring * np.cos(a), ring * np.sin(a), z])


def _golden_stride(N: int) -> int:
    target = N * (np.sqrt(5.0) - 1.0) / 2.0        # N / phi
    cands = [m for m in range(1, N + 1) if np.gcd(m, N) == 1]
    return min(cands, key=lambda m: (abs(m - target), m))


def initial(kind: str, d: int, k: int, N: int, s: float = 0.5) -> np.ndarray:
    if kind == "fibsphere":
        if k != 3:
            raise ValueError("the Fibonacci-sphere codebook is for k = 3")
        order = (np.arange(N) * _golden_stride(N)) % N
        return radii(d, 3, N)[:, None] * fibonacci_sphere(N)[order]
    u = directions(N, k, s)
    if kind == "sphere":
        return u
    return radii(d, k, N)[:, None] * u


def block_source(g: np.ndarray, k: int) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g[:, :k] / np.linalg.norm(g, axis=1, keepdims=True)


def _nearest(Y: np.ndarray, C: np.ndarray) -> tuple[np.ndarray, float]:
    n2 = np.einsum("ij,ij->i", C, C)
    idx = np.empty(len(Y), dtype=np.int64)
    err = 0.0
    rows = max(1, 8_000_000 // len(C))
    for a in range(0, len(Y), rows):
        y = Y[a:a + rows]
        score = y @ (-2.0 * C.T)
        score += n2
        i = score.argmin(axis=1)
        idx[a:a + rows] = i
        err += float(np.sum((y - C[i]) ** 2))
    return idx, err / len(Y)


def refine(C: np.ndarray, Y: np.ndarray, iters: int, rtol: float = 1e-6) -> tuple[np.ndarray, float]:
    C = C.copy()
    idx, mse = _nearest(Y, C)
    for _ in range(iters):
        cnt = np.bincount(idx, minlength=len(C)).astype(np.float64)
        tot = np.zeros_like(C)
        for j in range(C.shape[1]):
            tot[:, j] = np.bincount(idx, weights=Y[:, j], minlength=len(C))
        live = cnt > 0
        C[live] = tot[live] / cnt[live, None]
        idx, new = _nearest(Y, C)
        done = mse - new <= rtol * mse
        mse = new
        if done:
            break
    return C, mse


def build(kind: str, d: int, k: int, N: int, train_gaussians: np.ndarray, iters: int,
          restart_gaussians=(), s: float = 0.5) -> tuple[np.ndarray, float]:
    """(C fp64 [N, k], training MSE)."""
    Y = block_source(train_gaussians, k)
    C0 = initial(kind, d, k, N, s)
    best = refine(C0, Y, iters)
    for G in restart_gaussians:
        cand = refine(C0 @ haar(G).T, Y, iters)
        if cand[1] < best[1]:
            best = cand
    return best


def refine_gpu(C: np.ndarray, X, iters: int, rtol: float = 1e-6, device: int = 0) -> tuple[np.ndarray, float]:
    """``refine`` on the GPU. X: fp16 training rows [T, d] on the device; with the identity
    rotation every d/k block of a row, over the row's norm, is one draw of the block source. Each
    iteration is one library encode (the assignment: nearest codeword of every block) and one
    ``fq_centroid_sums`` (the centroid step); the distortion of the current codebook comes from the
    same sums: mean |u_b - c|^2 = (rows - 2 sum_n s_n.c_n + sum_n m_n |c_n|^2) / blocks."""
    import torch

    import random_access_kv_gb300 as fq
    C = np.array(C, dtype=np.float64, copy=True)
    N, k = C.shape
    T, d = X.shape
    eye = np.eye(d, dtype=np.float32)
    sums = torch.zeros((N, k), dtype=torch.float64, device=X.device)
    counts = torch.zeros(N, dtype=torch.float64, device=X.device)

    def assign(C):
        ctx = fq.fq_codebook_load(C.astype(np.float32), eye, device)
        nu, codes = fq.alloc_store(ctx, T, X.device)
        fq.fq_encode(ctx, X, T, nu, codes)
        sums.zero_()
        counts.zero_()
        fq.fq_centroid_sums(ctx, X, T, nu, codes, sums, counts)
        rows = float((nu > 0).sum().item())
        ctx.close()
        S, M = sums.cpu().numpy(), counts.cpu().numpy()
        Cf = C.astype(np.float32).astype(np.float64)      # the codebook the device searched
        mse = (rows - 2.0 * float(np.sum(S * Cf)) + float(np.sum(M * np.sum(Cf * Cf, axis=1)))) / (rows * (d // k))
        return S, M, mse

    S, M, mse = assign(C)
    for _ in range(iters):
        live = M > 0
        C[live] = S[live] / M[live, None]
        S, M, new = assign(C)
        done = mse - new <= rtol * mse
        mse = new
        if done:
            break
    return C, mse


def build_gpu(kind: str, d: int, k: int, N: int, train_rows, iters: int, restart_gaussians=(), s: float = 0.5,
              device: int = 0) -> tuple[np.ndarray, float]:
    """``build`` with the Lloyd iterations on the GPU (``refine_gpu``). train_rows: fp16 [T, d]
    rows (any array; copied to the device)."""
    import torch
    X = torch.as_tensor(np.ascontiguousarray(train_rows, dtype=np.float16)).to(f"cuda:{device}")
    C0 = initial(kind, d, k, N, s)
    best = refine_gpu(C0, X, iters, device=device)
    for G in restart_gaussians:
        cand = refine_gpu(C0 @ haar(G).T, X, iters, device=device)
        if cand[1] < best[1]:
            best = cand
    return best


def scalar_lloyd_max(d: int, N: int, tol: float = 1e-13, max_iter: int = 200000) -> tuple[np.ndarray, float]:
    """Scalar Lloyd-Max table for one coordinate y of a Haar-uniform unit d-vector: (levels
    ascending as C [N, 1], per-coordinate MSE). The density of y is proportional to
    (1 - y^2)^m, m = (d - 3)/2, on [-1, 1] (y^2 ~ Beta(1/2, (d - 1)/2)). Lloyd-Max alternates
    midpoint thresholds and cell centroids; cell masses use the regularised incomplete beta
    function and cell first moments the closed form of the integral of y (1 - y^2)^m. The density
    is log-concave, so the fixed point is unique."""
    if d < 3 or N < 1:
        raise ValueError("need d >= 3 and N >= 1")
    a, b = 0.5, 0.5 * (d - 1)
    m = 0.5 * (d - 3)
    norm = np.exp(special.betaln(a, b))           # integral of (1 - y^2)^m over [-1, 1]

    def half_mass(y):                             # P(0 <= Y <= |y|), without cancellation near 1
        return 0.5 * special.betainc(a, b, np.minimum(y * y, 1.0))

    def mass(lo, hi):
        both_pos, both_neg = lo >= 0, hi <= 0
        out = np.sign(hi) * half_mass(hi) - np.sign(lo) * half_mass(lo)
        # cells on one side: difference of upper-tail masses
        tail = lambda y: 0.5 * special.betaincc(a, b, np.minimum(y * y, 1.0))
        out = np.where(both_pos, tail(lo) - tail(hi), out)
        out = np.where(both_neg, tail(hi) - tail(lo), out)
        return out

    def moment(lo, hi):                           # integral of y f(y) over [lo, hi]
        return (np.power(1.0 - lo * lo, m + 1.0) - np.power(1.0 - hi * hi, m + 1.0)) / (2.0 * (m + 1.0) * norm)

    q = (np.arange(N, dtype=np.float64) + 0.5) / N
    c = np.sign(q - 0.5) * np.sqrt(special.betaincinv(a, b, np.abs(2.0 * q - 1.0)))
    for _ in range(max_iter):
        t = np.concatenate([[-1.0], 0.5 * (c[1:] + c[:-1]), [1.0]])
        P = mass(t[:-1], t[1:])
        new = moment(t[:-1], t[1:]) / P
        done = np.max(np.abs(new - c)) <= tol
        c = new
        if done:
            break
    t = np.concatenate([[-1.0], 0.5 * (c[1:] + c[:-1]), [1.0]])
    mse = 1.0 / d - float(np.sum(mass(t[:-1], t[1:]) * c * c))
    return c[:, None], mse


def for_workload(cfg: int) -> tuple[np.ndarray, np.ndarray]:
    """(C float32 [N, k], Pi float32 [d, d]) of one of the synthetic workloads."""
    import synth
    w = synth.WORKLOADS[cfg]
    Pi = haar(synth.rotation_gaussian(cfg, w.d)).astype(np.float32)
    C, _ = build(w.codebook_kind, w.d, w.k, w.N, synth.source_gaussians(cfg, w.lloyd_train, w.d),
                 w.lloyd_iters, [synth.restart_gaussian(cfg, w.k, r) for r in range(1, w.lloyd_restarts)],
                 synth.kronecker_offset(cfg))
    return C.astype(np.float32), Pi


# Codebook file (.fqb): the persistent state of a codec, i.e. the shared codebook and rotation with
# how they were built. Little-endian: a header, then C float32 [N x k] and Pi float32 [d x d] (row
# major), then the CRC-32 of everything before it.
FQB_MAGIC = b"FQB1"
FQB_VERSION = 1
_FQB_HEADER = struct.Struct("<4sIIII16sqIIQd")   # magic, version, d, k, N, kind, seed, iters, restarts, draws, mse


def save_fqb(path: str, C: np.ndarray, Pi: np.ndarray, kind: str, seed: int = 0, iters: int = 0,
             restarts: int = 0, draws: int = 0, mse: float = float("nan")) -> None:
    C = np.ascontiguousarray(C, dtype="<f4")
    Pi = np.ascontiguousarray(Pi, dtype="<f4")
    N, k = C.shape
    d = Pi.shape[0]
    if Pi.shape != (d, d):
        raise ValueError("Pi must be square")
    head = _FQB_HEADER.pack(FQB_MAGIC, FQB_VERSION, d, k, N, kind.encode()[:16].ljust(16, b"\0"), seed, iters,
                            restarts, draws, mse)
    body = head + C.tobytes() + Pi.tobytes()
    with open(path, "wb") as f:
        f.write(body + struct.pack("<I", zlib.crc32(body)))


def load_fqb(path: str) -> tuple[np.ndarray, np.ndarray, dict]:
    """(C float32 [N, k], Pi float32 [d, d], metadata). Raises ValueError on a damaged file."""
    with open(path, "rb") as f:
        data = f.read()
    if len(data) < _FQB_HEADER.size + 4:
        raise ValueError("fqb: truncated header")
    magic, version, d, k, N, kind, seed, iters, restarts, draws, mse = _FQB_HEADER.unpack_from(data)
    if magic != FQB_MAGIC or version != FQB_VERSION:
        raise ValueError("fqb: not a codebook file of this version")
    size = _FQB_HEADER.size + 4 * (N * k + d * d)
    if len(data) != size + 4:
        raise ValueError("fqb: size does not match the header")
    if struct.unpack_from("<I", data, size)[0] != zlib.crc32(data[:size]):
        raise ValueError("fqb: CRC mismatch")
    o = _FQB_HEADER.size
    C = np.frombuffer(data, dtype="<f4", count=N * k, offset=o).reshape(N, k).astype(np.float32)
    Pi = np.frombuffer(data, dtype="<f4", count=d * d, offset=o + 4 * N * k).reshape(d, d).astype(np.float32)
    meta = {"d": d, "k": k, "N": N, "kind": kind.rstrip(b"\0").decode(), "seed": seed, "lloyd_iters": iters,
            "restarts": restarts, "draws": draws, "mse": mse}
    return C, Pi, meta
