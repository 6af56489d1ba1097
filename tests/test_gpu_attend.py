"""Fused decode-into-attention (fq_attend) against the oracle's fp64 attention over the decoded
cache: every block layout (d/k = 1, 8, 16, 32, 64, 128), the score-table and direct-dot score forms,
long sequences split over a CTA cluster, ragged token counts, several queries per cached group,
gapped and interleaved row layouts, peaked softmax, and the argument checks."""
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


_CTX = {}

# (d, k, N, source): a workload's codebook and rotation, or a seeded random codebook ("rand").
SHAPES = [(64, 2, 16, 1), (64, 2, 256, 2), (64, 4, 1024, 3), (128, 8, 4096, 4), (64, 64, 4096, 5),
          (64, 8, 512, "rand"), (128, 2, 64, "rand"), (128, 4, 256, "rand"), (64, 1, 256, "rand"),
          (128, 1, 64, "rand"), (64, 4, 4096, "rand"), (128, 2, 8192, "rand")]


def tables(d, k, N, src):
    key = (d, k, N, src)
    if key not in _CTX:
        if src == "rand":
            r = np.random.default_rng([d, k, N])
            C = (r.standard_normal((N, k)) / np.sqrt(d)).astype(np.float32)
            Pi = ocb.haar_rotation(r.standard_normal((d, d))).astype(np.float32)
        else:
            C, Pi = ow.codebook(src), ow.rotation(src)
        _CTX[key] = (fq.fq_codebook_load(C, Pi), C, Pi)
    return _CTX[key]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_case(shape, G, T, k_row0, v_row0, stride, qpg=1, scale=None, sub=0):
    d, k, N, src = shape
    ctx, C, Pi = tables(*shape)
    nb, B = d // k, int(np.log2(N))
    M = max(k_row0, v_row0) + (G - 1) * stride + T + 3
    nw = fq.fq_code_words(ctx, M)
    nu, words = synth.random_store(d * 1000 + k, M, nw, sub)
    q = synth.query_rows(d, G * qpg, d, sub)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out = torch.full((G * qpg, d), np.nan, dtype=torch.float32, device="cuda")
    fq.fq_attend(ctx, dev(nu), dev(words.view(np.int32)), M, dev(q), G * qpg, qpg, T, k_row0, v_row0,
                 stride, scale, out)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    got = out.cpu().numpy()
    worst = 0.0
    for g in range(G):
        kr, vr = k_row0 + g * stride, v_row0 + g * stride
        worst = max(worst, parity.check_attention(
            got[g * qpg:(g + 1) * qpg], q[g * qpg:(g + 1) * qpg].astype(np.float64),
            nu[kr:kr + T], ofq.record_range(words, kr, T, nb, B),
            nu[vr:vr + T], ofq.record_range(words, vr, T, nb, B), C, Pi, scale))
    return worst


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"d{s[0]}k{s[1]}N{s[2]}")
@pytest.mark.parametrize("T", [1, 33, 300])
def test_attend_gapped_layout(shape, T):
    # keys of all groups first, then values; rows of consecutive groups 5 apart beyond T
    G, stride = 5, T + 5
    run_case(shape, G, T, 7, 7 + G * stride, stride)


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[2], SHAPES[3], SHAPES[4]], ids=lambda s: f"d{s[0]}k{s[1]}")
def test_attend_interleaved_long_split(shape):
    # two groups of 5000 tokens, key and value blocks of a group adjacent: the launch splits each
    # query over a cluster of CTAs
    T = 5000
    run_case(shape, 2, T, 0, T, 2 * T, sub=1)


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[2], SHAPES[3], SHAPES[4], SHAPES[5], SHAPES[8]],
                         ids=lambda s: f"d{s[0]}k{s[1]}N{s[2]}")
@pytest.mark.parametrize("qpg", [2, 4, 8])
def test_attend_several_queries_per_group(shape, qpg):
    # q_per_group a multiple of 4: clusters serve four queries of a group together, sharing the
    # decode; otherwise one query per cluster
    run_case(shape, 3, 130, 0, 3 * 130, 130, qpg=qpg, sub=2)


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[3]], ids=lambda s: f"d{s[0]}k{s[1]}")
def test_attend_grouped_queries_long_split(shape):
    # four queries per group over 5000 tokens: grouped clusters split over several CTAs
    T = 5000
    run_case(shape, 2, T, 0, T, 2 * T, qpg=4, sub=4)


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[4]], ids=lambda s: f"d{s[0]}k{s[1]}")
def test_attend_peaked_softmax(shape):
    # a large score scale concentrates the softmax on a few tokens
    run_case(shape, 4, 257, 0, 4 * 257, 257, scale=3.0, sub=3)


def test_attend_argument_checks():
    ctx, _, _ = tables(64, 2, 256, 2)
    M = 100
    nu = torch.ones(M, device="cuda")
    codes = torch.zeros(fq.fq_code_words(ctx, M), dtype=torch.int32, device="cuda")
    q = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    out = torch.zeros((2, 64), device="cuda")
    fq.fq_attend(ctx, nu, codes, M, q, 0, 1, 10, 0, 50, 10, 0.1, out)      # no queries: no-op
    for args in [(2, 1, 0, 0, 50, 10),     # T = 0
                 (2, 1, 10, 0, 95, 10),    # value rows beyond M
                 (2, 1, 10, 0, 50, 45),    # second group's values beyond M
                 (2, 3, 10, 0, 50, 10),    # queries not a multiple of the group size
                 (2, 1, 10, -1, 50, 10)]:  # negative row
        with pytest.raises(fq.FQError) as e:
            fq.fq_attend(ctx, nu, codes, M, q, *args, 0.1, out)
        assert e.value.code == 1
    with pytest.raises(fq.FQError):
        fq.fq_attend(ctx, nu, codes, M, q, 2, 1, 10, 0, 50, 10, float("inf"), out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
