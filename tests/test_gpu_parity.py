"""Parity of the CUDA path (through the C ABI) with the oracle, at sizes the oracle finishes in
seconds: several 128-row tiles plus a ragged tail, every workload's codebook and rotation, and the
edge cases (empty, single row, zero and non-finite rows, out-of-range gathers, records that
straddle words, appends into a partly filled store)."""
import numpy as np
import pytest

import parity
import synth
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


def ctx_for(cfg):
    if cfg not in _CTX:
        _CTX[cfg] = (fq.fq_codebook_load(ow.codebook(cfg), ow.rotation(cfg)), ow.codebook(cfg), ow.rotation(cfg))
    return _CTX[cfg]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_encode(ctx, x, row0=0, rows=None, fill=None):
    M = x.shape[0]
    rows = row0 + M if rows is None else rows
    nu = torch.zeros(max(rows, 1), dtype=torch.float32, device="cuda")
    nw = max(1, fq.fq_code_words(ctx, rows))
    if fill is None:
        codes = torch.zeros(nw, dtype=torch.int32, device="cuda")
    else:
        codes = dev(np.asarray(fill[:nw]).view(np.int32))
    fq.fq_encode(ctx, dev(x) if M else None, M, nu, codes, row0)
    torch.cuda.synchronize()
    return nu, codes


def gpu_gather(ctx, nu, codes, M, idx, d, f32=False):
    n = len(idx)
    out = torch.empty((max(n, 1), d), dtype=torch.float32 if f32 else torch.float16, device="cuda")
    fn = fq.fq_decode_gather_f32 if f32 else fq.fq_decode_gather
    fn(ctx, nu, codes, M, dev(np.asarray(idx, dtype=np.int64)), n, out)
    torch.cuda.synchronize()
    return out[:n].cpu().numpy()


REDUCED_ROWS = {1: 4096, 2: 128 * 37 + 45, 3: 128 * 37 + 45, 4: 128 * 11 + 92, 5: 128 * 15 + 61}


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_encode_decode_parity(cfg):
    ctx, C, Pi = ctx_for(cfg)
    w = synth.WORKLOADS[cfg]
    M = REDUCED_ROWS[cfg]
    x = synth.kv_tensor(cfg, 0, rows=M)
    nu_d, codes_d = gpu_encode(ctx, x)
    words = codes_d.cpu().numpy().view(np.uint32)
    nb = w.d // w.k
    idx_gpu = ofq.unpack(words, M, nb, w.B)
    agree, nmis, worst, nu_orc = parity.check_indices(x, C, Pi, idx_gpu)
    parity.check_nu(nu_d.cpu().numpy()[:M], nu_orc)
    parity.check_packing(words, idx_gpu, w.B)
    # full decode (fp16) and gathers (fp16 and fp32) of the device's own codes
    out = torch.empty((M, w.d), dtype=torch.float16, device="cuda")
    fq.fq_decode(ctx, nu_d, codes_d, M, out)
    torch.cuda.synchronize()
    nu_g = nu_d.cpu().numpy()[:M].astype(np.float64)
    parity.check_decode(out.cpu().numpy(), nu_g, idx_gpu, C, Pi, fp16_output=True)
    sel = synth.gather_indices(cfg, 0, M, 777)
    g32 = gpu_gather(ctx, nu_d, codes_d, M, sel, w.d, f32=True)
    parity.check_decode(g32, nu_g[sel], idx_gpu[sel], C, Pi, fp16_output=False)
    g16 = gpu_gather(ctx, nu_d, codes_d, M, sel, w.d)
    parity.check_decode(g16, nu_g[sel], idx_gpu[sel], C, Pi, fp16_output=True)
    assert fq.fq_status(ctx) == 0


@pytest.mark.parametrize("M", [1, 31, 127, 128, 129, 1000])
def test_ragged_sizes(M):
    ctx, C, Pi = ctx_for(2)
    x = synth.gaussian_rows(2, 0, M, 64, scale_spread=True)
    nu_d, codes_d = gpu_encode(ctx, x)
    words = codes_d.cpu().numpy().view(np.uint32)
    idx = ofq.unpack(words, M, 32, 8)
    _, _, _, nu_orc = parity.check_indices(x, C, Pi, idx)
    parity.check_nu(nu_d.cpu().numpy()[:M], nu_orc)
    parity.check_packing(words, idx, 8)


def test_empty_calls_are_no_ops():
    ctx, _, _ = ctx_for(2)
    nu = torch.full((4,), 7.0, device="cuda")
    codes = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    fq.fq_encode(ctx, None, 0, nu, codes, 0)
    fq.fq_decode_gather(ctx, nu, codes, 1, None, 0, None)
    fq.fq_decode(ctx, nu, codes, 0, None)
    torch.cuda.synchronize()
    assert torch.all(nu == 7.0) and torch.all(codes == -1)


def test_zero_and_non_finite_rows():
    ctx, C, Pi = ctx_for(2)
    x = synth.gaussian_rows(2, 1, 300, 64)
    x[5] = 0
    x[100, 3] = np.float16(np.inf)
    x[200, 7] = np.float16(np.nan)
    nu_d, codes_d = gpu_encode(ctx, x)
    assert fq.fq_status(ctx) & fq.FQ_FLAG_NONFINITE
    assert fq.fq_status(ctx) == 0                        # the flag was cleared by the read
    nu = nu_d.cpu().numpy()
    words = codes_d.cpu().numpy().view(np.uint32)
    idx = ofq.unpack(words, 300, 32, 8)
    for r in (5, 100, 200):
        assert nu[r] == 0 and not idx[r].any()
    keep = np.setdiff1d(np.arange(300), [100, 200])
    parity.check_indices(x[keep], C, Pi, idx[keep])
    out = gpu_gather(ctx, nu_d, codes_d, 300, [5, 100], 64)
    assert not out.any()


def test_gather_out_of_range_rows_are_zero_and_flagged():
    ctx, C, Pi = ctx_for(2)
    x = synth.gaussian_rows(2, 2, 200, 64)
    nu_d, codes_d = gpu_encode(ctx, x)
    assert fq.fq_status(ctx) == 0
    sel = np.array([3, -1, 199, 200, 10 ** 12, 0])
    out = gpu_gather(ctx, nu_d, codes_d, 200, sel, 64, f32=True)
    assert fq.fq_status(ctx) & fq.FQ_FLAG_RANGE
    assert not out[[1, 3, 4]].any()
    idx = ofq.unpack(codes_d.cpu().numpy().view(np.uint32), 200, 32, 8)
    ok = [0, 2, 5]
    parity.check_decode(out[ok], nu_d.cpu().numpy()[sel[ok]], idx[sel[ok]], C, Pi, fp16_output=False)


@pytest.mark.parametrize("f32", [False, True])
def test_d128_gather_many_tiles_per_cta_with_out_of_range_rows(f32):
    # The d = 128 decoder pipelines consecutive tiles of a CTA through two A buffers and two
    # accumulators: 152 x 6 tiles plus a ragged tail give every CTA six or seven tiles, so that
    # every buffer is reused and every barrier phase wraps. Repeated and out-of-range indices mixed
    # in; rows are checked against the oracle on a sample and out-of-range rows must be zero.
    ctx, C, Pi = ctx_for(4)
    M = 2000
    x = synth.gaussian_rows(4, 9, M, 128, scale_spread=True)
    nu_d, codes_d = gpu_encode(ctx, x)
    assert fq.fq_status(ctx) == 0
    n = 152 * 6 * 128 + 77
    r = np.random.default_rng(5)
    sel = r.integers(0, M, size=n)
    bad = r.choice(n, size=300, replace=False)
    sel[bad[:100]] = -1 - r.integers(0, 50, size=100)
    sel[bad[100:]] = M + r.integers(0, 10 ** 9, size=200)
    out = gpu_gather(ctx, nu_d, codes_d, M, sel, 128, f32=f32)
    assert fq.fq_status(ctx) & fq.FQ_FLAG_RANGE
    assert not out[bad].any()
    idx_all = ofq.unpack(codes_d.cpu().numpy().view(np.uint32), M, 16, 12)
    nu = nu_d.cpu().numpy()
    good = np.setdiff1d(np.arange(n), bad)
    pick = np.concatenate([good[:300], good[-300:], r.choice(good, size=1400, replace=False)])
    parity.check_decode(out[pick], nu[sel[pick]], idx_all[sel[pick]], C, Pi, fp16_output=not f32)


def _small_codebook(d, k, N, seed):
    from oracle import codebook as ocb
    r = np.random.default_rng(seed)
    Pi = ocb.haar_rotation(r.standard_normal((d, d))).astype(np.float32)
    if k == d:
        C = ocb.kronecker_directions(N, k, 0.37) * r.uniform(0.5, 1.0, size=(N, 1))
    elif k == 3:
        C = ocb.initial_codebook("fibsphere", d, 3, N)
    else:
        C = ocb.companded_radii(d, k, N)[:, None] * ocb.kronecker_directions(N, k, 0.5) if k >= 3 else \
            (ocb.spiral_codebook(d, N) if k == 2 else np.sort(r.standard_normal((N, 1)) * 0.2, axis=0))
    return C.astype(np.float32), Pi


@pytest.mark.parametrize("d,k,N", [(64, 4, 8), (64, 8, 2), (64, 2, 2), (128, 1, 8), (64, 64, 128),
                                   (128, 4, 64), (64, 1, 16), (64, 4, 256), (128, 8, 128), (64, 8, 512),
                                   (128, 4, 1024), (128, 2, 64), (64, 2, 128), (64, 1, 2), (128, 1, 4),
                                   (128, 2, 256), (64, 8, 4096), (128, 8, 4096),
                                   (96, 3, 8), (96, 3, 64), (96, 3, 512), (96, 3, 4096), (96, 1, 4),
                                   (96, 2, 16), (96, 4, 256), (96, 8, 128)])
@pytest.mark.parametrize("row0", [0, 1, 7, 45])
def test_records_at_any_bit_offset_preserve_neighbours(d, k, N, row0):
    C, Pi = _small_codebook(d, k, N, d * 1000 + k * 10 + N)
    ctx = fq.fq_codebook_load(C, Pi)
    R = fq.fq_record_bits(ctx)
    assert R == (d // k) * int(np.log2(N))
    M, tail = 333, 5
    rows = row0 + M + tail
    x = synth.gaussian_rows(7, 0, M, d, scale_spread=True)
    fill = np.random.default_rng(row0).integers(0, 2 ** 32, size=fq.fq_code_words(ctx, rows) + 1, dtype=np.uint64).astype(np.uint32)
    nu_d, codes_d = gpu_encode(ctx, x, row0=row0, rows=rows, fill=fill)
    words = codes_d.cpu().numpy().view(np.uint32)
    before = np.unpackbits(fill[:words.size].view(np.uint8), bitorder="little")
    after = np.unpackbits(words.view(np.uint8), bitorder="little")
    lo, hi = row0 * R, (row0 + M) * R
    np.testing.assert_array_equal(after[:lo], before[:lo])
    np.testing.assert_array_equal(after[hi:], before[hi:])
    idx = np.array([ofq.record_indices(words, row0 + m, d // k, int(np.log2(N))) for m in range(M)])
    _, _, _, nu_orc = parity.check_indices(x, C, Pi, idx)
    parity.check_nu(nu_d.cpu().numpy()[row0:row0 + M], nu_orc)
    got = gpu_gather(ctx, nu_d, codes_d, rows, np.arange(row0, row0 + M), d, f32=True)
    parity.check_decode(got, nu_d.cpu().numpy()[row0:row0 + M], idx, C, Pi, fp16_output=False)
    ctx.close()


@pytest.mark.parametrize("n", [1, 127, 129])
@pytest.mark.parametrize("f32", [False, True])
def test_d128_gather_of_few_rows(n, f32):
    # One CTA (one tile: the second builder group has none) and one row either side of a tile.
    ctx, C, Pi = ctx_for(4)
    M = 300
    x = synth.gaussian_rows(4, 10, M, 128, scale_spread=True)
    nu_d, codes_d = gpu_encode(ctx, x)
    sel = np.random.default_rng(n).integers(0, M, size=n)
    got = gpu_gather(ctx, nu_d, codes_d, M, sel, 128, f32=f32)
    idx = ofq.unpack(codes_d.cpu().numpy().view(np.uint32), M, 16, 12)
    parity.check_decode(got, nu_d.cpu().numpy()[sel], idx[sel], C, Pi, fp16_output=not f32)
    assert fq.fq_status(ctx) == 0


@pytest.mark.parametrize("d,k,N", [(128, 1, 8), (128, 2, 256), (128, 4, 64), (128, 8, 128)])
def test_d128_fp16_gather_with_run_time_field_widths(d, k, N):
    # The d = 128 decoder's fp16 output path (staged rows, TMA box stores) for every k, with
    # records whose fields are read at run time, over several tiles and a ragged tail.
    C, Pi = _small_codebook(d, k, N, d * 7 + k * 3 + N)
    ctx = fq.fq_codebook_load(C, Pi)
    M = 1500
    x = synth.gaussian_rows(7, 1, M, d, scale_spread=True)
    nu_d, codes_d = gpu_encode(ctx, x)
    sel = np.random.default_rng(k).integers(0, M, size=128 * 5 + 37)
    got = gpu_gather(ctx, nu_d, codes_d, M, sel, d)
    words = codes_d.cpu().numpy().view(np.uint32)
    B = int(np.log2(N))
    idx = np.array([ofq.record_indices(words, int(r), d // k, B) for r in sel])
    parity.check_decode(got, nu_d.cpu().numpy()[sel], idx, C, Pi, fp16_output=True)
    assert fq.fq_status(ctx) == 0
    ctx.close()


def test_append_matches_per_sequence_encode():
    ctx, C, Pi = ctx_for(4)
    n_seq, n_new, cap, t0 = 3, 50, 200, 17
    x = synth.gaussian_rows(4, 3, n_seq * n_new, 128, scale_spread=True)
    rows = n_seq * cap
    nu = torch.zeros(rows, device="cuda")
    codes = torch.zeros(fq.fq_code_words(ctx, rows), dtype=torch.int32, device="cuda")
    fq.fq_encode_append(ctx, dev(x), n_seq, n_new, cap, t0, nu, codes)
    nu2 = torch.zeros(rows, device="cuda")
    codes2 = torch.zeros_like(codes)
    for s in range(n_seq):
        fq.fq_encode(ctx, dev(x[s * n_new:(s + 1) * n_new]), n_new, nu2, codes2, s * cap + t0)
    torch.cuda.synchronize()
    assert torch.equal(codes, codes2) and torch.equal(nu, nu2)
    with pytest.raises(fq.FQError):
        fq.fq_encode_append(ctx, dev(x), n_seq, n_new, cap, cap - n_new + 1, nu, codes)


def test_misaligned_buffers_are_rejected():
    ctx, _, _ = ctx_for(2)
    x = torch.zeros(65 * 64, dtype=torch.float16, device="cuda")
    nu, codes = fq.alloc_store(ctx, 64)
    with pytest.raises(fq.FQError) as e:
        fq.fq_encode(ctx, x.data_ptr() + 2, 64, nu, codes)
    assert e.value.code == 4
    with pytest.raises(fq.FQError) as e:
        fq.fq_encode(ctx, x, -1, nu, codes)
    assert e.value.code == 1
