"""fp64 oracle of the FibQuant encoder and decoder (TEST INFRASTRUCTURE ONLY; see package header).

Each function restates one step of [FibQuant §2.3] in plain numpy, without blocking or fusion
beyond memory-bounded chunking of independent rows.

Conventions (the page leaves them open; readings listed in the design notes):
  * row form: x is a row of X [M, d]; u = Pi x / nu is computed as U = X Pi^T / nu.
  * a zero row has nu = 0, every index 0, and decodes to zero (Theorem 1 covers nonzero inputs).
  * ties in the nearest-codeword search go to the lowest codeword index.
  * record m occupies bits [m R, m R + R) of a little-endian stream of 32-bit words, LSB first;
    block b's index occupies bits [m R + b B, m R + b B + B), B = log2 N, R = (d / k) B.
"""
from __future__ import annotations

import math

import numpy as np


def bits_per_index(N: int) -> int:
    """B = log2 N; N must be a power of two [FibQuant §2.3, rate b = log2(N) / k]."""
    B = int(round(math.log2(N)))
    if N < 2 or (1 << B) != N:
        raise ValueError("N must be a power of two >= 2")
    return B


def record_bits(d: int, k: int, N: int) -> int:
    """R = (d / k) log2 N bits per vector, i.e. b = log2(N) / k bits per coordinate [FibQuant §2.3]."""
    if d % k:
        raise ValueError("k must divide d")
    return (d // k) * bits_per_index(N)


def row_norms(x) -> np.ndarray:
    """nu = ||x||_2 per row, in fp64 [FibQuant §2.3, encoder]."""
    x = np.asarray(x, dtype=np.float64)
    return np.sqrt(np.sum(x * x, axis=1))


def rotate_normalise(x, Pi, nu) -> np.ndarray:
    """u = Pi x / nu per row, fp64 [FibQuant §2.1 and §2.3]. Rows with nu = 0 give u = 0."""
    x = np.asarray(x, dtype=np.float64)
    Pi = np.asarray(Pi, dtype=np.float64)
    nu = np.asarray(nu, dtype=np.float64)
    y = x @ Pi.T
    u = np.zeros_like(y)
    nz = nu > 0
    u[nz] = y[nz] / nu[nz, None]
    return u


def split_blocks(u, k: int) -> np.ndarray:
    """The d / k consecutive blocks of size k of each row: [M, d] -> [M, d/k, k] [FibQuant §2.3]."""
    M, d = u.shape
    if d % k:
        raise ValueError("k must divide d")
    return u.reshape(M, d // k, k)


def nearest_codeword(points, C, chunk_elems: int = 1 << 23) -> np.ndarray:
    """argmin_n sum_j (p_j - c_nj)^2 for each point p (rows of ``points`` [n, k]) against C [N, k].

    Distances are formed from direct differences, in fp64. numpy's argmin returns the first
    minimum, so exact ties go to the lowest index [FibQuant §2.3, nearest-codeword lookup]."""
    P = np.asarray(points, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    n, k = P.shape
    N = C.shape[0]
    out = np.empty(n, dtype=np.int64)
    step = max(1, chunk_elems // (N * k))
    for s in range(0, n, step):
        diff = P[s:s + step, None, :] - C[None, :, :]
        out[s:s + step] = np.argmin(np.sum(diff * diff, axis=2), axis=1)
    return out


def encode(x, C, Pi) -> tuple[np.ndarray, np.ndarray]:
    """Encoder [FibQuant §2.3]: nu = ||x||, u = Pi x / nu, split into d/k blocks, nearest codeword
    per block. Returns (nu fp64 [M], indices int64 [M, d/k])."""
    C = np.asarray(C, dtype=np.float64)
    k = C.shape[1]
    nu = row_norms(x)
    u = rotate_normalise(x, Pi, nu)
    blocks = split_blocks(u, k)
    M, nb, _ = blocks.shape
    idx = nearest_codeword(blocks.reshape(M * nb, k), C).reshape(M, nb)
    idx[nu == 0] = 0
    return nu, idx


def decode(nu, idx, C, Pi) -> np.ndarray:
    """Decoder [FibQuant §2.3]: fetch the codewords, concatenate the blocks, apply the inverse
    rotation Pi^T and scale by the norm: x_hat = nu Pi^T concat(c_{i_b}). Row form:
    X_hat = nu * (Y_hat Pi). Returns fp64 [M, d]."""
    C = np.asarray(C, dtype=np.float64)
    Pi = np.asarray(Pi, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    M, nb = idx.shape
    yhat = C[idx].reshape(M, nb * C.shape[1])
    return np.asarray(nu, dtype=np.float64)[:, None] * (yhat @ Pi)


def pack(idx, B: int) -> np.ndarray:
    """Fixed-address packing [FibQuant §1 (fixed addresses, no variable-length codes) and §2.3]:
    record m at bit m R of an LSB-first stream, block b's index at bit m R + b B. Unused bits of
    the last 32-bit word are zero. Returns uint32 words."""
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= (1 << B)):
        raise ValueError("index out of range")
    bits = ((idx[..., None] >> np.arange(B)) & 1).astype(np.uint64).reshape(-1)
    nwords = (bits.size + 31) // 32
    padded = np.zeros(nwords * 32, dtype=np.uint64)
    padded[:bits.size] = bits
    words = np.sum(padded.reshape(nwords, 32) << np.arange(32, dtype=np.uint64), axis=1)
    return words.astype(np.uint32)


def unpack(words, M: int, nb: int, B: int) -> np.ndarray:
    """Inverse of ``pack`` for the first M records: [M, nb] int64 indices [FibQuant §2.3]."""
    words = np.asarray(words, dtype=np.uint32).astype(np.uint64)
    bits = ((words[:, None] >> np.arange(32, dtype=np.uint64)) & 1).reshape(-1)
    need = M * nb * B
    if bits.size < need:
        raise ValueError("too few words")
    b = bits[:need].reshape(M, nb, B).astype(np.int64)
    return np.sum(b << np.arange(B), axis=2)


def record_range(words, m0: int, count: int, nb: int, B: int) -> np.ndarray:
    """Indices [count, nb] of the consecutive records m0 .. m0 + count - 1, read from their fixed
    addresses (record m starts at bit m R) [FibQuant §1, §2.3]."""
    R = nb * B
    lo, hi = m0 * R, (m0 + count) * R
    w = np.asarray(words, dtype=np.uint32)[lo // 32:(hi + 31) // 32].astype(np.uint64)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint64)) & 1).reshape(-1)
    b = bits[lo % 32:lo % 32 + count * R].reshape(count, nb, B).astype(np.int64)
    return np.sum(b << np.arange(B), axis=2)


def record_indices(words, m: int, nb: int, B: int) -> np.ndarray:
    """Indices of the single record m, read bit by bit from its fixed address m R: the random
    access that the fixed-rate layout allows [FibQuant §1]."""
    words = np.asarray(words, dtype=np.uint32)
    R = nb * B
    out = np.zeros(nb, dtype=np.int64)
    for b in range(nb):
        v = 0
        for t in range(B):
            pos = m * R + b * B + t
            v |= int((int(words[pos // 32]) >> (pos % 32)) & 1) << t
        out[b] = v
    return out
