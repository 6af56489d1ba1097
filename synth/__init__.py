"""Seeded synthetic inputs for the FibQuant codec: KV tensors, random draws, workload table.

This module holds no arithmetic of the codec itself. It only draws random numbers with a fixed
recipe and names the five workloads (shapes, block size k, codebook size N, codebook-building
budgets). Everything the method computes from these draws (the Haar rotation from a Gaussian
matrix, codebook radii and directions, Lloyd refinement, encode and decode) lives elsewhere:
once in the oracle and once, independently, in the library.

The workloads stand in for the KV caches the FibQuant page evaluates on (GPT-2 small and
TinyLlama-1.1B, "FibQuant: universal vector quantisation for random-access KV-cache compression",
sections 4.2 and 4.3). No model weights or text are used: keys and values are drawn from the
distributions described per workload below.

Random streams: ``rng(cfg, stream, *sub)`` is ``numpy.random.default_rng([cfg, stream, *sub])``.
Stream 0 = K data, 1 = V data, 2 = the Gaussian matrix behind the rotation, 3 = codebook
building (Lloyd training draws, restart rotations, Kronecker offset), 4 = gather indices,
5 = attention queries, 6 = random code stores, 7 = symbol streams for the iterated-map archive.

The archive workloads (``ARCHIVE_WORKLOADS``) stand in for the inputs of the page "Fractal KV-Cache
Archives" (gist.science summary of arXiv 2607.07144), whose codec timings are quoted on a document
of a million characters: a byte stream with a text-like skew, and the index streams of a KV cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

STREAM_K, STREAM_V, STREAM_ROT, STREAM_CODEBOOK, STREAM_GATHER = 0, 1, 2, 3, 4
STREAM_QUERY, STREAM_STORE, STREAM_SYMBOLS = 5, 6, 7


def rng(cfg: int, stream: int, *sub: int) -> np.random.Generator:
    return np.random.default_rng([int(cfg), int(stream), *[int(s) for s in sub]])


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: KV tensor shape, codec parameters and codebook-building budget."""

    cfg: int
    name: str
    shape: tuple            # per-tensor shape, last dim = d; rows = prod(shape[:-1])
    tensors: int            # 1 (a single X) or 2 (K and V)
    k: int
    N: int
    data: str               # "gauss", "channel_scaled", "token_lognormal"
    codebook_kind: str      # "spiral" (k=2), "kronecker" (k>=3), "sphere" (k=d unit directions)
    lloyd_train: int        # training draws from the spherical-Beta source
    lloyd_iters: int
    lloyd_restarts: int
    op: str                 # "encode+decode", "encode+gather", "stream+gather"
    gather: int = 0         # gathered rows per tensor (encode+gather) or token positions (stream+gather)
    stream_new: int = 0     # new tokens per sequence per append step (stream+gather)
    extra: dict = field(default_factory=dict)

    @property
    def d(self) -> int:
        return int(self.shape[-1])

    @property
    def rows(self) -> int:
        return int(np.prod(self.shape[:-1]))

    @property
    def B(self) -> int:
        return int(round(math.log2(self.N)))


# The five workloads. Lloyd budgets other than workload 1's five iterations are chosen here (the
# pages fix none): they bound codebook-building time on the host.
WORKLOADS = {
    1: Workload(1, "tiny: 4096x64 N(0,1), k=2 N=16 (b=2)", (4096, 64), 1, 2, 16, "gauss", "spiral",
                4096, 5, 1, "encode+decode"),
    2: Workload(2, "GPT-2-small KV 12x12x1024x64, k=2 N=256 (b=4)", (12, 12, 1024, 64), 2, 2, 256,
                "channel_scaled", "spiral", 65536, 20, 4, "encode+gather", gather=65536),
    3: Workload(3, "TinyLlama KV 22x8x4x4096x64, k=4 N=1024 (b=2.5)", (22, 8, 4, 4096, 64), 2, 4, 1024,
                "channel_scaled", "kronecker", 131072, 10, 2, "encode+decode"),
    4: Workload(4, "Llama long-context KV 32x8x32768x128, k=8 N=4096 (b=1.5)", (32, 8, 32768, 128), 2, 8,
                4096, "token_lognormal", "kronecker", 65536, 6, 2, "stream+gather",
                gather=3277, stream_new=1024),
    5: Workload(5, "GPT-2 KV 12x12x1024x64, k=d=64 N=4096 (b=0.1875)", (12, 12, 1024, 64), 2, 64, 4096,
                "gauss", "sphere", 32768, 6, 2, "encode+decode"),
}


def _channel_scaled(r: np.random.Generator, shape, out: np.ndarray) -> None:
    """z ~ N(0,1) times a per-(layer, head, channel) scale exp(U[ln .5, ln 8]); one channel per
    (layer, head) (round(0.02 d) = 1 for d = 64) is multiplied by 20. For a 5-D (L, B, H, T, d)
    shape the batch axis shares its layer's scales."""
    d = shape[-1]
    if len(shape) == 4:
        L, H, T = shape[0], shape[1], shape[2]
        Bt = 1
    else:
        L, Bt, H, T = shape[0], shape[1], shape[2], shape[3]
    n_out = max(1, int(round(0.02 * d)))
    scale = np.exp(r.uniform(math.log(0.5), math.log(8.0), size=(L, H, d)))
    for l in range(L):
        for h in range(H):
            ch = r.choice(d, size=n_out, replace=False)
            scale[l, h, ch] *= 20.0
    o = out.reshape(L, Bt, H, T, d)
    for l in range(L):
        z = r.standard_normal((Bt, H, T, d), dtype=np.float32)
        z *= scale[l][None, :, None, :].astype(np.float32)
        o[l] = z.astype(np.float16)


def _token_lognormal(r: np.random.Generator, shape, out: np.ndarray) -> None:
    """x = s_t z with z ~ N(0, I_d) and s_t ~ LogNormal(0, 0.5) per (layer, head, token)."""
    L, H, T, d = shape
    o = out.reshape(L, H, T, d)
    for l in range(L):
        s = r.lognormal(0.0, 0.5, size=(H, T, 1)).astype(np.float32)
        z = r.standard_normal((H, T, d), dtype=np.float32)
        z *= s
        o[l] = z.astype(np.float16)


def kv_tensor(cfg: int, which: int = 0, rows: int | None = None) -> np.ndarray:
    """Tensor ``which`` (0 = K or the single X, 1 = V) of workload ``cfg`` as fp16 [rows, d].

    ``rows`` truncates to the first rows (the draw order is fixed, so a prefix is the same
    prefix of the full tensor only for the plain Gaussian workloads; for the scaled ones the
    prefix is drawn from the first layer's scales). Values are rounded to fp16 with
    round-to-nearest-even (numpy's cast)."""
    w = WORKLOADS[cfg]
    r = rng(cfg, STREAM_K if which == 0 else STREAM_V)
    if w.data == "gauss":
        n = w.rows if rows is None else min(rows, w.rows)
        return r.standard_normal((n, w.d), dtype=np.float32).astype(np.float16)
    if w.data == "token_lognormal":
        # Layers are drawn one after another, so a prefix needs only its first layers drawn.
        per_layer = int(np.prod(w.shape[1:-1]))
        n_layers = w.shape[0] if rows is None else min(w.shape[0], -(-rows // per_layer))
        shape = (n_layers,) + tuple(w.shape[1:])
        out = np.empty((n_layers * per_layer, w.d), dtype=np.float16)
        _token_lognormal(r, shape, out)
        return out if rows is None or rows >= out.shape[0] else out[:rows].copy()
    out = np.empty((w.rows, w.d), dtype=np.float16)
    if w.data == "channel_scaled":
        _channel_scaled(r, w.shape, out)
    else:
        raise ValueError(w.data)
    return out if rows is None else out[:rows].copy()


def gaussian_rows(cfg: int, which: int, rows: int, d: int, scale_spread: bool = False) -> np.ndarray:
    """A small fp16 [rows, d] Gaussian tensor with the workload's seed, for reduced-size cases.
    With ``scale_spread`` the rows get lognormal(0, 0.5) norms and one column is multiplied by 20
    (an outlier channel), so that reduced cases keep the heavy-tailed structure."""
    r = rng(cfg, 10 + which, rows, d)
    z = r.standard_normal((rows, d), dtype=np.float32)
    if scale_spread:
        z *= r.lognormal(0.0, 0.5, size=(rows, 1)).astype(np.float32)
        z[:, int(r.integers(d))] *= 20.0
    return z.astype(np.float16)


def rotation_gaussian(cfg: int, d: int, draw: int = 0) -> np.ndarray:
    """d x d standard Gaussian (fp64) from which the shared rotation is built by QR."""
    return rng(cfg, STREAM_ROT, draw).standard_normal((d, d))


def source_gaussians(cfg: int, T: int, d: int, chunk: int = 0) -> np.ndarray:
    """T x d standard Gaussian draws (fp64); the spherical-Beta training points are their first k
    coordinates divided by the row norm."""
    return rng(cfg, STREAM_CODEBOOK, 0, chunk).standard_normal((T, d))


def restart_gaussian(cfg: int, k: int, restart: int) -> np.ndarray:
    """k x k Gaussian behind the seeded rotation of the codebook initialisation for restart r >= 1."""
    return rng(cfg, STREAM_CODEBOOK, 1, restart).standard_normal((k, k))


def kronecker_offset(cfg: int) -> float:
    """Offset s of the Roberts-Kronecker sequence: 1/2 for workloads 3 and 4, a seeded U(0,1)
    draw for the k = d workload 5."""
    if WORKLOADS[cfg].codebook_kind == "sphere":
        return float(rng(cfg, STREAM_CODEBOOK, 2).uniform())
    return 0.5


def gather_indices(cfg: int, which: int, M: int, n: int, replace: bool = True) -> np.ndarray:
    """n row indices in [0, M) as int64, uniform with replacement (default) or without."""
    r = rng(cfg, STREAM_GATHER, which)
    if replace:
        return r.integers(0, M, size=n, dtype=np.int64)
    return r.choice(M, size=n, replace=False).astype(np.int64)


def token_positions(cfg: int, T: int, n: int) -> np.ndarray:
    """n distinct token positions in [0, T), random order (shared by all layers and heads)."""
    return rng(cfg, STREAM_GATHER, 9).permutation(T)[:n].astype(np.int64)


def query_rows(cfg: int, n: int, d: int, sub: int = 0) -> np.ndarray:
    """Attention queries: n fp16 rows [n, d] of N(0, 1) entries (stream 5)."""
    return rng(cfg, STREAM_QUERY, sub).standard_normal((n, d)).astype(np.float16)


def random_store(cfg: int, M: int, n_words: int, sub: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """A code store of M rows with uniformly random bits and log-normal norms (stream 6):
    (nu float32 [M], words uint32 [n_words]). With N a power of two every bit pattern is a valid
    record, so this exercises all codewords without running an encoder. Norms are
    exp(N(log 8, 0.5^2)), about the norm of a 64-dimensional row of unit-variance entries."""
    r = rng(cfg, STREAM_STORE, sub)
    nu = np.exp(r.normal(np.log(8.0), 0.5, size=M)).astype(np.float32)
    words = r.integers(0, 1 << 32, size=n_words, dtype=np.uint64).astype(np.uint32)
    return nu, words


@dataclass(frozen=True)
class ArchiveWorkload:
    """Symbol streams for the iterated-map archive: n_streams streams of T symbols over N."""

    name: str
    n_streams: int
    T: int
    N: int
    law: str            # "zipf": p(c) proportional to (c + 1)^-1.1; "uniform"
    append: int         # symbols per stream per append call in the streaming measurement
    lookups: int        # random-access positions per step


ARCHIVE_WORKLOADS = {
    "document": ArchiveWorkload("document: 1 stream of 2^20 bytes, N=256, Zipf(1.1)", 1, 1 << 20, 256, "zipf",
                                1, 1 << 20),
    "kv-streams": ArchiveWorkload("KV index streams: 144 (layer, head) streams x 1024 tokens x 32 indices, N=256",
                                  144, 32768, 256, "uniform", 32, 1 << 20),
}


def symbol_streams(n_streams: int, T: int, N: int, law: str = "uniform", sub: int = 0) -> np.ndarray:
    """uint16 [n_streams, T] symbols in [0, N) (stream 7). ``zipf`` draws symbol c with probability
    proportional to (c + 1)^-1.1, the skew of characters in text; ``uniform`` suits codec indices,
    which a well-built codebook makes close to equiprobable."""
    r = rng(N, STREAM_SYMBOLS, n_streams, T, sub)
    if law == "uniform":
        return r.integers(0, N, size=(n_streams, T), dtype=np.int64).astype(np.uint16)
    if law == "zipf":
        p = 1.0 / np.arange(1, N + 1, dtype=np.float64) ** 1.1
        return r.choice(N, size=(n_streams, T), p=p / p.sum()).astype(np.uint16)
    raise ValueError(law)


def stream_positions(n_streams: int, T_cap: int, T: int, n: int, sub: int = 0) -> np.ndarray:
    """n flat positions q T_cap + t (stream q < n_streams, position t < T), uniform (stream 7)."""
    r = rng(n_streams, STREAM_SYMBOLS, T, n, 1000 + sub)
    return r.integers(0, n_streams, size=n) * int(T_cap) + r.integers(0, T, size=n)
