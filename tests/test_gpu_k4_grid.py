"""The k = 4 candidate-grid encoder against the oracle on inputs aimed at its weak points: blocks
placed within about 1e-4 of the midpoint of two neighbouring codewords (near ties, where the
listed candidates must include both), blocks on codewords, blocks far outside the grid (one
coordinate near 1, the exhaustive fallback), rows mixing all of these with Gaussian rows, and the
smallest and largest codebooks the encoder takes (N = 2 and N = 4096), at d = 64 and d = 128.
Indices must agree with the oracle's nearest codeword (near ties excepted), records must be
bit-exact repacks of the indices, and nu within its tolerance."""
import numpy as np
import pytest

import parity
import synth
from oracle import codebook as ocb
from oracle import fibquant as ofq
from oracle import workloads as ow

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import random_access_kv_gb300 as fq  # noqa: E402
from random_access_kv_gb300 import build as fbuild  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _encode(ctx, x):
    M = x.shape[0]
    nu = torch.zeros(M, dtype=torch.float32, device="cuda")
    codes = torch.zeros(max(1, fq.fq_code_words(ctx, M)), dtype=torch.int32, device="cuda")
    fq.fq_encode(ctx, torch.from_numpy(np.ascontiguousarray(x)).cuda(), M, nu, codes, 0)
    torch.cuda.synchronize()
    return nu.cpu().numpy(), codes.cpu().numpy().view(np.uint32), fq.fq_status(ctx)


def _rows_at(u_blocks, Pi, scale, d):
    """fp16 rows whose normalised rotation has the given leading blocks: the last block is set so
    that the whole vector has unit norm (u = x Pi^T / |x|, so x = u Pi)."""
    M, nb, k = u_blocks.shape
    u = np.zeros((M, d))
    u[:, :nb * k] = u_blocks.reshape(M, -1)
    rest = 1.0 - np.sum(u * u, axis=1)
    assert (rest > 0).all()
    u[:, d - 1] = np.sqrt(rest)
    x = (u @ np.asarray(Pi, dtype=np.float64)) * scale[:, None]
    return x.astype(np.float16)


def _adversarial_rows(C, Pi, d, seed, M=1024):
    r = np.random.default_rng(seed)
    C64 = np.asarray(C, dtype=np.float64)
    N, k = C64.shape
    nb = d // k // 2                     # leading blocks placed; the last coordinate fixes the norm
    scale = np.exp(r.normal(0.0, 0.5, M))
    # Midpoints of a codeword and its nearest neighbour, scaled into the unit ball's share.
    d2 = np.sum((C64[:, None, :] - C64[None, :, :]) ** 2, axis=2)
    np.fill_diagonal(d2, np.inf)
    nn = np.argmin(d2, axis=1)
    pick = r.integers(0, N, size=(M, nb))
    mid = 0.5 * (C64[pick] + C64[nn[pick]]) + r.normal(0.0, 1e-4, size=(M, nb, k))
    at = C64[r.integers(0, N, size=(M, nb))]
    blocks = np.where((np.arange(M) % 2 == 0)[:, None, None], mid, at)
    # The rare row whose placed blocks hold more than 0.95 of a unit vector's energy is shrunk
    # (its blocks then leave the midpoints; they remain valid test points).
    e = np.sum(blocks.reshape(M, -1) ** 2, axis=1)
    blocks = blocks / np.sqrt(np.maximum(1.0, e / 0.95))[:, None, None]
    x = _rows_at(blocks, Pi, scale, d)
    # Spikes: almost all energy in one rotated coordinate (outside the grid).
    spikes = np.zeros((64, d))
    spikes[np.arange(64), r.integers(0, d, 64)] = 1.0
    spikes += r.normal(0.0, 0.02, size=spikes.shape)
    xs = (spikes @ np.asarray(Pi, dtype=np.float64)).astype(np.float16)
    xg = synth.gaussian_rows(3, 5, 333, d, scale_spread=True)
    bad = synth.gaussian_rows(3, 6, 2, d)
    bad[0, 3] = np.float16(np.nan)
    bad[1, d - 1] = np.float16(np.inf)
    # The last five rows: three zero rows, then a NaN row and an Inf row.
    return np.concatenate([x, xs, xg, np.zeros((3, d), np.float16), bad])


def _random_codebook(N, d, seed):
    r = np.random.default_rng(seed)
    C = r.standard_normal((N, 4)) / np.sqrt(d)
    Pi = ocb.haar_rotation(r.standard_normal((d, d)))
    return C.astype(np.float32), Pi.astype(np.float32)


CASES = {
    "w3-codebook": lambda: (ow.codebook(3), ow.rotation(3), 64),
    "N4096-d64": lambda: (*_random_codebook(4096, 64, 11), 64),
    "N256-d128": lambda: (*_random_codebook(256, 128, 12), 128),
    "N2-d64": lambda: (*_random_codebook(2, 64, 13), 64),
    "N1024-d128": lambda: (*_random_codebook(1024, 128, 14), 128),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_grid_encoder_matches_the_oracle_on_adversarial_rows(case):
    C, Pi, d = CASES[case]()
    ctx = fq.fq_codebook_load(C, Pi)
    try:
        x = _adversarial_rows(C, Pi, d, seed=len(case))
        nu, words, status = _encode(ctx, x)
        assert status == fq.FQ_FLAG_NONFINITE
        B = int(np.log2(C.shape[0]))
        idx = np.array([ofq.record_indices(words, m, d // 4, B) for m in range(x.shape[0])])
        parity.check_packing(words, idx, B)
        assert (idx[-5:] == 0).all() and (nu[-5:] == 0).all()
        fin = x.shape[0] - 2
        # Near ties are the point of these rows, so more indices than usual may differ; every
        # difference must still be a near tie.
        _, nmis, worst, nu_orc = parity.check_indices(x[:fin], C, Pi, idx[:fin], agreement=0.99)
        parity.check_nu(nu[:fin], nu_orc)
    finally:
        ctx.close()
