"""fp64 oracle of the contractive iterated-map archive of a symbol stream (TEST INFRASTRUCTURE ONLY).

Source: the page "Fractal KV-Cache Archives" (gist.science summary of arXiv 2607.07144), cited as
[Archive §x]. It proposes storing the index stream a vector quantiser produces as points of the plane:

  * [Archive §Method 1, mechanism] a regular N-gon is fixed with one vertex V(c) per symbol c of the
    alphabet {0 .. N-1}; symbol c_k moves the current point by the contraction
        p_k = V(c_k) + r (p_{k-1} - V(c_k)),   0 < r < 1 the contraction ratio.
  * [Archive §Method 1, properties] the map is invertible (lossless) when r is small enough that the
    symbols' cells are disjoint; encoding takes linear time; a position is read back by rebuilding
    only the stretch it needs from the nearest stored anchor point.
  * [Archive §Method 1, implementation] to keep floating-point error from growing during inversion,
    one point is stored per fixed-length segment, and the segment is rebuilt from it by an anchored
    backward search.

Readings of what the page leaves open (each restated in the design notes):
  * V(c) = (cos(2 pi c / N), sin(2 pi c / N)): the N-gon inscribed in the unit circle, vertex 0 on
    the positive x axis, counter-clockwise.
  * Every segment starts at the centre of the polygon (the origin), so segments are independent;
    the stored anchor of a segment is its last point. Segment s of a stream holds positions
    [s L, s L + L); the last segment may hold fewer. A batch of streams of capacity T_cap keeps
    ceil(T_cap / L) anchors per stream.
  * The cell of symbol c is the image of the unit disc under its map: the disc of radius r about
    (1 - r) V(c). Adjacent centres are 2 (1 - r) sin(pi / N) apart, so the cells are disjoint
    exactly when r < sin(pi / N) / (1 + sin(pi / N)).
  * The backward search: at each step the symbol is the one whose cell centre is nearest to the
    current point (ties to the lowest index), after which its map is inverted,
    p_{k-1} = V(c) + (p_k - V(c)) / r.
  * Arithmetic is fp64 with every operation rounded, in the order written above (no fused
    multiply-add): t = p - V, t = r t, p = V + t, per coordinate. r is the fp64 number given.
  * The segment length is the largest L for which a worst-case bound on the rounding error of the
    forward steps, amplified by 1/r per backward step, stays below half the margin between a cell
    and the edge of its angular sector (``max_segment``).

Parity status: vertices, ratio_limit, encode, decode, access and append are pinned in
tests/test_oracle_fractal.py (closed forms, a 40-digit evaluation of the unrolled recurrence,
exhaustive round trips of every short string, adversarial strings at the segment-length limit,
failure beyond it, the suffix-distance identity). The segment-length bound is this module's own
derivation, pinned by those round trips.
"""
from __future__ import annotations

import math

import numpy as np

U = 2.0 ** -53          # unit roundoff of fp64


def vertices(N: int) -> np.ndarray:
    """V [N, 2]: the regular N-gon on the unit circle, vertex c at angle 2 pi c / N [Archive §Method 1]."""
    if N < 2:
        raise ValueError("the alphabet needs at least two symbols")
    c = np.arange(N, dtype=np.float64)
    a = 2.0 * np.pi * c / N
    return np.stack([np.cos(a), np.sin(a)], axis=1)


def ratio_limit(N: int) -> float:
    """Largest contraction ratio with disjoint cells: sin(pi/N) / (1 + sin(pi/N)) (strict bound)."""
    s = math.sin(math.pi / N)
    return s / (1.0 + s)


def cell_margin(N: int, r: float) -> float:
    """Distance from every cell to the edges of its angular sector: (1 - r) sin(pi/N) - r.

    The disc of radius r about (1 - r) V(c) lies between the two rays at angles 2 pi c / N +- pi / N
    with at least this much room; a point closer to its cell than that is decided correctly."""
    return (1.0 - r) * math.sin(math.pi / N) - r


def max_segment(N: int, r: float, cap: int = 64) -> int:
    """Largest segment length whose backward search is exact in fp64, by a worst-case error bound.

    Forward step, per coordinate: t = p - V, t = r t, p = V + t with |p| <= 1 and |p - V| <= 2
    commits an error below delta = 1.01 u (1 + 4 r). A backward step commits at most eta = 8 u
    (this module divides by r; a kernel may multiply by a rounded 1/r with a fused multiply-add).
    If e_k is the error of the rebuilt point against the stored forward point at step k, then
    e_{k-1} <= (e_k + delta) / r + eta, and e_L = 0 at the anchor, so after j backward steps
    |e| <= sqrt(2) (delta + r eta) r^-j / (1 - r) (Euclidean). The L decisions of a segment
    use j = 0 .. L-1, so every one is correct when that bound at j = L - 1 is at most half the cell
    margin. Returns that largest L, at most ``cap``; 0 when not even one symbol fits (or r is not
    below the disjointness limit)."""
    if not (0.0 < r < ratio_limit(N)):
        return 0
    g = cell_margin(N, r)
    delta = 1.01 * U * (1.0 + 4.0 * r)
    eta = 8.0 * U
    amp = math.sqrt(2.0) * (delta + r * eta) / (1.0 - r)
    if amp > 0.5 * g:
        return 0
    # largest j with amp r^-j <= g / 2, then L = j + 1
    j = int(math.floor(math.log(0.5 * g / amp) / math.log(1.0 / r)))
    while j >= 0 and amp * (1.0 / r) ** j > 0.5 * g:    # guard the floor against log rounding
        j -= 1
    return min(cap, j + 1)


def encode_segment(symbols, N: int, r: float, start=(0.0, 0.0), V=None) -> tuple[float, float]:
    """The point after applying the maps of ``symbols`` in order to ``start`` [Archive §Method 1].

    Plain Python floats (IEEE fp64, every operation rounded), one symbol at a time."""
    if V is None:
        V = vertices(N)
    x, y = float(start[0]), float(start[1])
    r = float(r)
    for c in symbols:
        c = int(c)
        if not 0 <= c < N:
            raise ValueError(f"symbol {c} is outside the alphabet of {N}")
        vx, vy = float(V[c, 0]), float(V[c, 1])
        x = vx + r * (x - vx)
        y = vy + r * (y - vy)
    return x, y


def segments(T_cap: int, L: int) -> int:
    """Anchors kept per stream of capacity T_cap: ceil(T_cap / L)."""
    return -(-int(T_cap) // int(L))


def encode(symbols, N: int, r: float, L: int, T_cap: int | None = None) -> np.ndarray:
    """Anchors [n_streams, ceil(T_cap / L), 2] of the streams ``symbols`` [n_streams, T] (or [T]).

    Segment s of a stream is encoded from the origin over positions [s L, min(s L + L, T)); its
    anchor is the last point [Archive §Method 1, implementation]. Anchors of segments beyond T are
    left at the origin."""
    sym = np.atleast_2d(np.asarray(symbols, dtype=np.int64))
    n_streams, T = sym.shape
    T_cap = T if T_cap is None else int(T_cap)
    if T > T_cap:
        raise ValueError("more symbols than the capacity")
    V = vertices(N)
    S = segments(T_cap, L)
    out = np.zeros((n_streams, S, 2), dtype=np.float64)
    for q in range(n_streams):
        for s in range(segments(T, L)):
            out[q, s] = encode_segment(sym[q, s * L:min(s * L + L, T)], N, r, V=V)
    return out


def append(anchors, T_old: int, new, N: int, r: float, L: int) -> np.ndarray:
    """Anchors after appending ``new`` [n_streams, n] symbols to streams holding T_old symbols.

    The partial last segment continues from its stored point; later segments start at the origin.
    The result equals ``encode`` of the whole streams [Archive §Method 1, linear-time encoding]."""
    A = np.array(anchors, dtype=np.float64, copy=True)
    new = np.atleast_2d(np.asarray(new, dtype=np.int64))
    n_streams, n = new.shape
    V = vertices(N)
    if (T_old + n) > A.shape[1] * L:
        raise ValueError("the appended symbols do not fit the streams' capacity")
    for q in range(n_streams):
        t = 0
        while t < n:
            pos = T_old + t
            s, off = divmod(pos, L)
            take = min(L - off, n - t)
            start = tuple(A[q, s]) if off else (0.0, 0.0)
            A[q, s] = encode_segment(new[q, t:t + take], N, r, start=start, V=V)
            t += take
    return A


def nearest_cell(x: float, y: float, N: int, r: float, V=None) -> int:
    """Symbol whose cell centre (1 - r) V(c) is nearest to (x, y); ties to the lowest index."""
    if V is None:
        V = vertices(N)
    cx, cy = (1.0 - r) * V[:, 0], (1.0 - r) * V[:, 1]
    return int(np.argmin((x - cx) ** 2 + (y - cy) ** 2))


def decode_segment(anchor, length: int, N: int, r: float, stop: int = 0, V=None) -> list[int]:
    """Symbols of positions [stop, length) of a segment, rebuilt backward from its anchor.

    At each step the symbol is the nearest cell's; the map of that symbol is then inverted
    [Archive §Method 1, anchored backward search]. Returned in position order."""
    if V is None:
        V = vertices(N)
    x, y = float(anchor[0]), float(anchor[1])
    r = float(r)
    out = []
    for k in range(length - 1, stop - 1, -1):
        c = nearest_cell(x, y, N, r, V)
        out.append(c)
        if k > stop:
            vx, vy = float(V[c, 0]), float(V[c, 1])
            x = vx + (x - vx) / r
            y = vy + (y - vy) / r
    return out[::-1]


def segment_length(T: int, L: int, s: int) -> int:
    """Symbols held by segment s of a stream of T symbols."""
    return max(0, min(L, T - s * L))


def decode(anchors, T: int, N: int, r: float, L: int) -> np.ndarray:
    """All T symbols of every stream [n_streams, T] from their anchors."""
    A = np.asarray(anchors, dtype=np.float64)
    V = vertices(N)
    out = np.zeros((A.shape[0], T), dtype=np.int64)
    for q in range(A.shape[0]):
        for s in range(segments(T, L)):
            n = segment_length(T, L, s)
            out[q, s * L:s * L + n] = decode_segment(A[q, s], n, N, r, V=V)
    return out


def access(anchors, T: int, N: int, r: float, L: int, stream: int, t: int) -> int:
    """The symbol at position t of a stream: backward from its segment's anchor to position t only
    [Archive §Method 1, random access from the nearest anchor]."""
    if not 0 <= t < T:
        raise IndexError("position outside the stream")
    s, off = divmod(int(t), L)
    A = np.asarray(anchors, dtype=np.float64)
    return decode_segment(A[stream, s], segment_length(T, L, s), N, r, stop=off)[0]
