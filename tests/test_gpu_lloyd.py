"""Codebook Lloyd iterations on the GPU (assignment by the library's encoder, centroids by
fq_centroid_sums) against the oracle's Lloyd iteration on the same training blocks."""
import numpy as np
import pytest

from oracle import codebook as ocb
from random_access_kv_gb300 import codebook as pcb

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import random_access_kv_gb300 as fq  # noqa: E402
from random_access_kv_gb300 import build as fbuild  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def blocks(X16, k):
    """The training draws the GPU sees: every k-block of each fp16 row over the row's norm."""
    X = X16.astype(np.float64)
    U = X / np.linalg.norm(X, axis=1, keepdims=True)
    return U.reshape(-1, k)


@pytest.mark.parametrize("kind,d,k,N", [("spiral", 64, 2, 256), ("kronecker", 64, 4, 1024), ("kronecker", 128, 8, 512),
                                        ("kronecker", 64, 1, 16), ("sphere", 64, 64, 256)], ids=lambda v: str(v))
def test_one_lloyd_step_matches_the_oracle(kind, d, k, N):
    """One Lloyd step [FibQuant §2.2, refinement]: the assignment (the library's encoder, identity
    rotation) against the oracle's nearest-codeword rule, and the centroid step (fq_centroid_sums)
    against the oracle's centroids of the same assignment."""
    from oracle import fibquant as ofq
    import parity
    r = np.random.default_rng([d, k, N])
    X16 = r.standard_normal((3000 if k < d else 40000, d)).astype(np.float16)
    C0 = ocb.initial_codebook(kind, d, k, N, 0.37 if k == d else 0.5)
    C0f = C0.astype(np.float32)
    eye = np.eye(d, dtype=np.float32)
    T = X16.shape[0]
    # Assignment: every block index is the oracle's, or a near tie of it (distance gap within the
    # codec's 1e-5 relative rule).
    ctx = fq.fq_codebook_load(C0f, eye)
    X = torch.from_numpy(X16).cuda()
    nu, codes = fq.alloc_store(ctx, T)
    fq.fq_encode(ctx, X, T, nu, codes)
    sums = torch.zeros((N, k), dtype=torch.float64, device="cuda")
    counts = torch.zeros(N, dtype=torch.float64, device="cuda")
    fq.fq_centroid_sums(ctx, X, T, nu, codes, sums, counts)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    ctx.close()
    idx_gpu = ofq.unpack(codes.cpu().numpy().view(np.uint32), T, d // k, int(np.log2(N)))
    parity.check_indices(X16, C0f, eye, idx_gpu)
    # Centroid step: the oracle's sums over the device's own assignment. Counts are exact; every
    # centroid agrees to the fp32 accuracy of the device's block coordinates (u = x / nu in fp32,
    # relative error below 1e-7, so an average of them errs by less than 1e-6).
    Y = blocks(X16, k)
    a = idx_gpu.reshape(-1)
    cnt_orc = np.bincount(a, minlength=N).astype(np.float64)
    sum_orc = np.stack([np.bincount(a, weights=Y[:, j], minlength=N) for j in range(k)], axis=1)
    S, M = sums.cpu().numpy(), counts.cpu().numpy()
    np.testing.assert_array_equal(M, cnt_orc)
    live = M > 0
    np.testing.assert_allclose(S[live] / M[live, None], sum_orc[live] / cnt_orc[live, None], rtol=0, atol=1e-6)
    # The whole step through the GPU builder: the oracle's Lloyd step lands on the same
    # distortion (a near tie moves one block between two cells, which changes the MSE by far less).
    C1_orc, hist = ocb.lloyd(C0, Y, iters=1, tol=0.0)
    C1_gpu, mse1 = pcb.refine_gpu(C0, X, iters=1, rtol=0.0)
    assert mse1 == pytest.approx(hist[-1], rel=1e-4)
    # Codewords whose cells hold the same blocks on both sides move to the same centroid.
    a_orc = ocb.assign(Y, C0)
    same = np.array([np.array_equal(np.flatnonzero(a == n), np.flatnonzero(a_orc == n)) for n in range(N)])
    np.testing.assert_allclose(C1_gpu[same], C1_orc[same], rtol=0, atol=1e-6)


def test_gpu_build_reaches_the_host_builders_distortion():
    d, k, N = 64, 2, 64
    r = np.random.default_rng(9)
    X16 = r.standard_normal((40000, d)).astype(np.float16)
    C_gpu, mse_gpu = pcb.build_gpu("spiral", d, k, N, X16, iters=15)
    C_host, mse_host = pcb.build("spiral", d, k, N, r.standard_normal((40000 * d // k, d)), 15)
    assert mse_gpu == pytest.approx(mse_host, rel=0.01)


def test_centroid_sums_argument_checks():
    C = ocb.spiral_codebook(64, 16).astype(np.float32)
    ctx = fq.fq_codebook_load(C, np.eye(64, dtype=np.float32))
    x = torch.zeros((10, 64), dtype=torch.float16, device="cuda")
    nu, codes = fq.alloc_store(ctx, 10)
    sums = torch.zeros((16, 2), dtype=torch.float64, device="cuda")
    counts = torch.zeros(16, dtype=torch.float64, device="cuda")
    fq.fq_centroid_sums(ctx, x, 0, nu, codes, sums, counts)        # no rows: no-op
    with pytest.raises(fq.FQError):
        fq.fq_centroid_sums(ctx, x, -1, nu, codes, sums, counts)
    fq.fq_encode(ctx, x, 10, nu, codes)
    fq.fq_centroid_sums(ctx, x, 10, nu, codes, sums, counts)       # zero rows are skipped
    torch.cuda.synchronize()
    assert float(counts.sum()) == 0.0 and float(sums.abs().sum()) == 0.0
    ctx.close()
