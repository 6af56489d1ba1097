"""A claim the page makes about rates, checked on the oracle: on the canonical spherical-Beta
source FibQuant has lower MSE than the scalar Lloyd-Max codec (k = 1) at every integer rate, and it
reaches rates between the integers [FibQuant §4.1 and the fractional rates of §4.3].

At b = 1 the k = 2 code has four points, and the best four-point code of the plane block is the
square that the scalar code already forms, so the gain there needs a larger block (k = 4, 16
codewords); from b = 2 on, k = 2 suffices."""
import numpy as np

from oracle import codebook as ocb
from oracle import fibquant as ofq
from random_access_kv_gb300 import codebook as pcb


def rel_mse(X, C, Pi):
    nu, idx = ofq.encode(X, C, Pi)
    Xh = ofq.decode(nu, idx, C, Pi)
    return float(np.mean(np.sum((X - Xh) ** 2, axis=1) / np.sum(X * X, axis=1)))


def test_vector_code_beats_scalar_table_at_integer_rates_and_fills_the_gaps():
    d = 64
    r = np.random.default_rng(5)
    Pi = ocb.haar_rotation(r.standard_normal((d, d)))
    X = r.standard_normal((3000, d)).astype(np.float16).astype(np.float64)
    Y = ocb.source_points(r.standard_normal((60_000, d)), 2)
    fib = {}
    for N in (4, 8, 16, 32, 64):                       # b = 1, 1.5, 2, 2.5, 3 at k = 2
        C, _ = ocb.build_codebook("spiral", d, 2, N, Y, iters=30)
        fib[np.log2(N) / 2] = rel_mse(X, C, Pi)
    Y4 = ocb.source_points(r.standard_normal((60_000, d)), 4)
    C4, _ = ocb.build_codebook("kronecker", d, 4, 16, Y4, iters=30)
    best = {1: rel_mse(X, C4, Pi), 2: fib[2.0], 3: fib[3.0]}
    for b in (1, 2, 3):
        C1, mse1 = pcb.scalar_lloyd_max(d, 2 ** b)
        scalar = rel_mse(X, C1, Pi)
        assert abs(scalar - d * mse1) < 0.05 * d * mse1   # the table's own MSE, estimated
        assert best[b] < 0.98 * scalar, (b, best[b], scalar)
    # fractional rates sit strictly between their integer neighbours
    assert fib[1.0] > fib[1.5] > fib[2.0] > fib[2.5] > fib[3.0]
