"""The scalar comparison codec (k = 1 with the exact Lloyd-Max table) and fractional-rate FibQuant
codebooks through the library: parity with the oracle, and the relative MSE the library delivers
equals the oracle's on the same rows."""
import numpy as np
import pytest

import parity
import synth
from oracle import codebook as ocb
from oracle import fibquant as ofq
from random_access_kv_gb300 import codebook as pcb

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import random_access_kv_gb300 as fq  # noqa: E402
from random_access_kv_gb300 import build as fbuild  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def codebook(kind, d, k, N):
    if kind == "scalar":
        return pcb.scalar_lloyd_max(d, N)[0].astype(np.float32)
    Y = ocb.source_points(np.random.default_rng([d, k, N]).standard_normal((16 * N + 4096, d)), k)
    return ocb.build_codebook(kind, d, k, N, Y, iters=8)[0].astype(np.float32)


@pytest.mark.parametrize("kind,d,k,N", [("scalar", 64, 1, 2), ("scalar", 64, 1, 16), ("scalar", 128, 1, 8),
                                        ("spiral", 64, 2, 32), ("spiral", 64, 2, 128),
                                        ("kronecker", 64, 4, 1024), ("kronecker", 128, 8, 256),
                                        ("fibsphere", 96, 3, 64), ("fibsphere", 96, 3, 512), ("scalar", 96, 1, 4)],
                         ids=lambda v: str(v))
def test_rate_point_parity_and_mse(kind, d, k, N):
    C = codebook(kind, d, k, N)
    Pi = ocb.haar_rotation(np.random.default_rng(d).standard_normal((d, d))).astype(np.float32)
    x = synth.gaussian_rows(1, 4, 1531, d)                       # several tiles and a ragged tail
    M = x.shape[0]
    ctx = fq.fq_codebook_load(C, Pi)
    nu, codes = fq.alloc_store(ctx, M)
    fq.fq_encode(ctx, torch.from_numpy(x).cuda(), M, nu, codes)
    out = torch.empty((M, d), dtype=torch.float32, device="cuda")
    fq.fq_decode_gather_f32(ctx, nu, codes, M, torch.arange(M, device="cuda"), M, out)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    words = codes.cpu().numpy().view(np.uint32)
    idx = ofq.unpack(words, M, d // k, int(np.log2(N)))
    agree, _, _, nu_orc = parity.check_indices(x, C, Pi, idx)
    parity.check_nu(nu.cpu().numpy(), nu_orc)
    parity.check_packing(words, idx, int(np.log2(N)))
    parity.check_decode(out.cpu().numpy(), nu.cpu().numpy(), idx, C, Pi, fp16_output=False)
    X = x.astype(np.float64)
    nu_o, idx_o = ofq.encode(X, C, Pi)
    mse_orc = np.mean(np.sum((X - ofq.decode(nu_o, idx_o, C, Pi)) ** 2, axis=1) / np.sum(X * X, axis=1))
    mse_lib = np.mean(np.sum((X - out.cpu().numpy()) ** 2, axis=1) / np.sum(X * X, axis=1))
    assert mse_lib == pytest.approx(mse_orc, rel=1e-3)
    ctx.close()
