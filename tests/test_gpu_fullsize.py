"""Full-size workloads, in the launch configuration the benchmark times (one call per tensor over all
rows), checked against the oracle on sampled rows, plus properties that hold at any size:
  * the encoder is row-independent, so streaming appends reproduce a one-shot encode bit for bit;
  * every norm is finite and non-negative and no device flag is raised.
"""
import numpy as np
import pytest

import parity
import synth
from oracle import fibquant as ofq
from oracle import workloads as ow

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import random_access_kv_gb300 as fq  # noqa: E402
from random_access_kv_gb300 import build as fbuild  # noqa: E402

SAMPLE = 1500


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def sampled_records(words, rows, nb, B):
    return np.array([ofq.record_indices(words, int(m), nb, B) for m in rows])


def check_sample(ctx, x, nu_d, codes_d, C, Pi, w, rows, M):
    words = codes_d.cpu().numpy().view(np.uint32)
    nb = w.d // w.k
    idx = sampled_records(words, rows, nb, w.B)
    nu_rows = nu_d.cpu().numpy()[rows]
    agree, nmis, worst, nu_orc = parity.check_indices(x[rows], C, Pi, idx)
    parity.check_nu(nu_rows, nu_orc)
    n = len(rows)
    for f32 in (True, False):
        out = torch.empty((n, w.d), dtype=torch.float32 if f32 else torch.float16, device="cuda")
        fn = fq.fq_decode_gather_f32 if f32 else fq.fq_decode_gather
        fn(ctx, nu_d, codes_d, M, torch.from_numpy(rows.astype(np.int64)).cuda(), n, out)
        torch.cuda.synchronize()
        parity.check_decode(out.cpu().numpy(), nu_rows, idx, C, Pi, fp16_output=not f32)
    return agree


@pytest.mark.parametrize("cfg,which", [(2, 0), (2, 1), (3, 0), (5, 0)])
def test_full_tensor_encode_and_decode(cfg, which):
    w = synth.WORKLOADS[cfg]
    C, Pi = ow.codebook(cfg), ow.rotation(cfg)
    ctx = fq.fq_codebook_load(C, Pi)
    x = synth.kv_tensor(cfg, which)
    M = x.shape[0]
    nu_d, codes_d = fq.alloc_store(ctx, M)
    fq.fq_encode(ctx, torch.from_numpy(x).cuda(), M, nu_d, codes_d)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    nu_all = nu_d.cpu().numpy()
    assert np.all(np.isfinite(nu_all)) and np.all(nu_all >= 0)
    rows = np.sort(synth.gather_indices(cfg, 7 + which, M, SAMPLE, replace=False))
    rows[0], rows[-1] = 0, M - 1                      # first and last record of the store
    check_sample(ctx, x, nu_d, codes_d, C, Pi, w, rows, M)
    if w.op == "encode+decode":
        # the benchmark's full decode, checked on the same sampled rows
        out = torch.empty((M, w.d), dtype=torch.float16, device="cuda")
        fq.fq_decode(ctx, nu_d, codes_d, M, out)
        torch.cuda.synchronize()
        words = codes_d.cpu().numpy().view(np.uint32)
        idx = sampled_records(words, rows, w.d // w.k, w.B)
        parity.check_decode(out[torch.from_numpy(rows).cuda()].cpu().numpy(), nu_all[rows], idx, C, Pi,
                            fp16_output=True)
    assert fq.fq_status(ctx) == 0
    ctx.close()


def test_streaming_append_long_context():
    """Workload 4: 32 append steps of 1024 new tokens into 256 (layer, head) sequences of capacity
    32768, then a gather of 10% of the token positions across all sequences."""
    cfg = 4
    w = synth.WORKLOADS[cfg]
    C, Pi = ow.codebook(cfg), ow.rotation(cfg)
    ctx = fq.fq_codebook_load(C, Pi)
    L, H, T, d = w.shape
    n_seq = L * H
    x = synth.kv_tensor(cfg, 0)                       # [L*H*T, d], sequences contiguous
    xs = x.reshape(n_seq, T, d)
    M = n_seq * T
    nu_d, codes_d = fq.alloc_store(ctx, M)
    for step in range(T // w.stream_new):
        t0 = step * w.stream_new
        chunk = np.ascontiguousarray(xs[:, t0:t0 + w.stream_new, :]).reshape(-1, d)
        fq.fq_encode_append(ctx, torch.from_numpy(chunk).cuda(), n_seq, w.stream_new, T, t0, nu_d, codes_d)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    # Row independence: the streamed store equals a one-shot encode of the whole tensor.
    nu2, codes2 = fq.alloc_store(ctx, M)
    fq.fq_encode(ctx, torch.from_numpy(x).cuda(), M, nu2, codes2)
    torch.cuda.synchronize()
    assert torch.equal(codes_d, codes2) and torch.equal(nu_d, nu2)
    del nu2, codes2
    # Random-access decode of 10% of the positions, shared by all sequences, in random order.
    pos = synth.token_positions(cfg, T, w.gather)
    gidx = (np.arange(n_seq)[:, None] * T + pos[None, :]).reshape(-1)
    n = len(gidx)
    out = torch.empty((n, d), dtype=torch.float16, device="cuda")
    fq.fq_decode_gather(ctx, nu_d, codes_d, M, torch.from_numpy(gidx).cuda(), n, out)
    torch.cuda.synchronize()
    sel = np.sort(synth.gather_indices(cfg, 8, n, SAMPLE, replace=False))
    rows = gidx[sel]
    words = codes_d.cpu().numpy().view(np.uint32)
    idx = sampled_records(words, rows, d // w.k, w.B)
    agree, _, _, nu_orc = parity.check_indices(x[rows], C, Pi, idx)
    parity.check_nu(nu_d[torch.from_numpy(rows).cuda()].cpu().numpy(), nu_orc)
    parity.check_decode(out[torch.from_numpy(sel).cuda()].cpu().numpy(),
                        nu_d[torch.from_numpy(rows).cuda()].cpu().numpy(), idx, C, Pi, fp16_output=True)
    assert fq.fq_status(ctx) == 0
    ctx.close()


@pytest.mark.parametrize("cfg,qpg", [(2, 1), (4, 1), (4, 4)])
def test_attend_full_size_sampled_groups(cfg, qpg):
    """Fused attention at the workload's full size, in the benchmark's launch configuration (keys at
    rows [0, M), values at [M, 2M), one group per (layer, head)), over a random store; sampled
    groups checked against the oracle's fp64 attention over the decoded records."""
    w = synth.WORKLOADS[cfg]
    C, Pi = ow.codebook(cfg), ow.rotation(cfg)
    ctx = fq.fq_codebook_load(C, Pi)
    T = int(w.shape[-2])
    groups = w.rows // T
    M = w.rows
    nb, B = w.d // w.k, w.B
    nu, words = synth.random_store(cfg, 2 * M, fq.fq_code_words(ctx, 2 * M), sub=7)
    q = synth.query_rows(cfg, groups * qpg, w.d, sub=7)
    scale = 1.0 / np.sqrt(w.d)
    out = torch.empty((groups * qpg, w.d), dtype=torch.float32, device="cuda")
    fq.fq_attend(ctx, torch.from_numpy(nu).cuda(), torch.from_numpy(words.view(np.int32)).cuda(), 2 * M,
                 torch.from_numpy(q).cuda(), groups * qpg, qpg, T, 0, M, T, scale, out)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for g in sorted({0, groups - 1} | set(synth.gather_indices(cfg, 9, groups, 2, replace=False).tolist())):
        kr, vr = g * T, M + g * T
        parity.check_attention(got[g * qpg:(g + 1) * qpg], q[g * qpg:(g + 1) * qpg].astype(np.float64),
                               nu[kr:kr + T], ofq.record_range(words, kr, T, nb, B),
                               nu[vr:vr + T], ofq.record_range(words, vr, T, nb, B), C, Pi, scale)
    ctx.close()
