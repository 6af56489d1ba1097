"""The iterated-map archive ("Fractal KV-Cache Archives", Method 1) through the C ABI, against the
oracle: anchors, full decode, random access, append, edge cases and device-side checks."""
import numpy as np
import pytest

import synth
from oracle import fractal as ofa

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import random_access_kv_gb300 as fq  # noqa: E402
from random_access_kv_gb300 import build as fbuild  # noqa: E402

from test_oracle_fractal import adversarial  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    fbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def to_dev(sym: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(sym, dtype=np.uint16).view(np.int16)).cuda()


def to_host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def make(N, rho=0.75, L=None):
    r = rho * ofa.ratio_limit(N)
    L = L or ofa.max_segment(N, r)
    return fq.fa_create(N, r, L), r, L


# Anchors: the library forms p = r (p - V) + V with one fused multiply-add, the oracle with a
# rounded product and a rounded sum. Per step and coordinate the two differ by at most
# delta_lib + delta_orc <= u (1 + 2r) + 1.01 u (1 + 4r) < 5.1 u (|p| <= 1, |p - V| <= 2, r < 1/2),
# and a difference made k steps before the end is scaled by r^k, so the sum over a segment is below
# 5.1 u / (1 - r) <= 10.2 u; one-ulp differences between the two vertex tables add at most u.
ANCHOR_TOL = 12 * 2.0 ** -53


def check_anchors(ctx, got, want):
    np.testing.assert_allclose(got, want, rtol=0, atol=ANCHOR_TOL)


def test_vertex_table_within_one_ulp_of_the_oracle():
    for N in (2, 3, 256, 4096):
        ctx, _, _ = make(N)
        V = fq.fa_vertex_table(ctx)
        np.testing.assert_allclose(V, ofa.vertices(N), rtol=0, atol=2 ** -53)
        assert fq.fa_params(ctx)[0] == N
        ctx.close()


@pytest.mark.parametrize("N,rho", [(2, 0.75), (3, 0.5), (16, 0.75), (256, 0.75), (256, 0.3), (1024, 0.75),
                                   (4096, 0.75)])
def test_encode_decode_access_parity(N, rho):
    ctx, r, L = make(N, rho)
    n_streams, T_cap, T = 3, 2003, 1997                 # several blocks of segments, ragged tails
    sym = synth.symbol_streams(n_streams, T, N, "uniform", sub=N)
    A = fq.alloc_archive(ctx, n_streams, T_cap)
    fq.fa_encode(ctx, to_dev(sym), n_streams, T, T_cap, 0, A)
    out = torch.empty((n_streams, T), dtype=torch.int16, device="cuda")
    fq.fa_decode(ctx, A, n_streams, T_cap, T, out)
    pos = synth.stream_positions(n_streams, T_cap, T, 5000, sub=N)
    pos = np.concatenate([pos, [0, T - 1, T_cap + L - 1, 2 * T_cap + min((T // L) * L, T - 1)]])   # segment edges
    acc = torch.empty(len(pos), dtype=torch.int16, device="cuda")
    fq.fa_access(ctx, A, n_streams, T_cap, T, torch.from_numpy(pos).cuda(), len(pos), acc)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == 0
    want = ofa.encode(sym, N, r, L, T_cap=T_cap)
    got = A.cpu().numpy()
    check_anchors(ctx, got, want)
    np.testing.assert_array_equal(to_host(out), sym)                           # lossless
    np.testing.assert_array_equal(to_host(acc), sym[pos // T_cap, pos % T_cap])
    # the oracle reads the library's anchors, and the library the oracle's
    q = 1
    np.testing.assert_array_equal(ofa.decode(got[q:q + 1], T, N, r, L)[0], sym[q])
    A2 = torch.from_numpy(want).cuda()
    fq.fa_decode(ctx, A2, n_streams, T_cap, T, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(out), sym)
    ctx.close()


def test_append_in_chunks_is_bit_identical_to_one_encode():
    N = 256
    ctx, r, L = make(N)
    n_streams, T_cap = 5, 300
    sym = synth.symbol_streams(n_streams, T_cap, N, "zipf", sub=1)
    A = fq.alloc_archive(ctx, n_streams, T_cap)
    fq.fa_encode(ctx, to_dev(sym), n_streams, T_cap, T_cap, 0, A)
    B = fq.alloc_archive(ctx, n_streams, T_cap)
    T = 0
    oracle_B = ofa.encode(sym[:, :0], N, r, L, T_cap=T_cap)
    for n in (1, 1, L - 2, 3, 2 * L + 1, 0, 100, T_cap - (1 + 1 + L - 2 + 3 + 2 * L + 1 + 100)):
        chunk = sym[:, T:T + n]
        fq.fa_encode(ctx, to_dev(chunk), n_streams, n, T_cap, T, B)
        oracle_B = ofa.append(oracle_B, T, chunk, N, r, L)
        T += n
    assert T == T_cap
    torch.cuda.synchronize()
    assert torch.equal(A, B)
    check_anchors(ctx, B.cpu().numpy(), oracle_B)
    ctx.close()


@pytest.mark.parametrize("N", [2, 4, 256, 4096])
def test_adversarial_strings_at_the_segment_limit(N):
    ctx, r, L = make(N)
    rng = np.random.default_rng(N)
    strings = adversarial(N, L, rng)                         # [64, L]: one stream per string
    n = strings.shape[0]
    A = fq.alloc_archive(ctx, n, L)
    fq.fa_encode(ctx, to_dev(strings), n, L, L, 0, A)
    out = torch.empty((n, L), dtype=torch.int16, device="cuda")
    fq.fa_decode(ctx, A, n, L, L, out)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == 0
    np.testing.assert_array_equal(to_host(out), strings)
    ctx.close()


def test_segment_lengths_below_the_limit_and_one():
    for L in (1, 2, 5):
        ctx, r, _ = make(64, 0.75, L)
        sym = synth.symbol_streams(2, 37, 64, sub=L)
        A = fq.alloc_archive(ctx, 2, 37)
        fq.fa_encode(ctx, to_dev(sym), 2, 37, 37, 0, A)
        out = torch.empty((2, 37), dtype=torch.int16, device="cuda")
        fq.fa_decode(ctx, A, 2, 37, 37, out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_host(out), sym)
        check_anchors(ctx, A.cpu().numpy(), ofa.encode(sym, 64, r, L))
        ctx.close()


def test_empty_calls_and_argument_checks():
    ctx, r, L = make(16)
    A = fq.alloc_archive(ctx, 2, 10)
    fq.fa_encode(ctx, None, 2, 0, 10, 0, A)                   # nothing to append
    fq.fa_decode(ctx, A, 2, 10, 0, None)                      # empty streams
    fq.fa_access(ctx, A, 2, 10, 5, None, 0, None)             # no lookups
    sym = to_dev(np.zeros((2, 4), np.uint16))
    for args in [(sym, 2, 4, 10, 7, A), (sym, -1, 4, 10, 0, A), (sym, 2, 4, 0, 0, A)]:
        with pytest.raises(fq.FQError):
            fq.fa_encode(ctx, *args)
    with pytest.raises(fq.FQError):
        fq.fa_decode(ctx, A, 2, 10, 11, torch.empty(22, dtype=torch.int16, device="cuda"))
    with pytest.raises(fq.FQError):                           # misaligned anchors
        fq.fa_encode(ctx, sym, 2, 4, 10, 0, A.view(-1)[1:].data_ptr())
    with pytest.raises(fq.FQError):
        fq.fa_create(16, r, L + 1)
    assert fq.fa_segments(ctx, 10) == -(-10 // L)
    ctx.close()


def test_device_checks_flag_bad_symbols_positions_and_anchors():
    N = 16
    ctx, r, L = make(N)
    sym = synth.symbol_streams(1, 3 * L, N, sub=2)
    sym[0, L + 1] = N                                         # outside the alphabet: segment 1 poisoned
    A = fq.alloc_archive(ctx, 1, 3 * L)
    fq.fa_encode(ctx, to_dev(sym), 1, 3 * L, 3 * L, 0, A)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == fq.FA_FLAG_SYMBOL
    a = A.cpu().numpy()
    assert np.isnan(a[0, 1]).all() and np.isfinite(a[0, [0, 2]]).all()
    out = torch.empty((1, 3 * L), dtype=torch.int16, device="cuda")
    fq.fa_decode(ctx, A, 1, 3 * L, 3 * L, out)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == fq.FA_FLAG_CORRUPT
    o = to_host(out)[0]
    assert np.all(o[L:2 * L] == 0xFFFF)
    np.testing.assert_array_equal(o[:L], sym[0, :L])
    np.testing.assert_array_equal(o[2 * L:], sym[0, 2 * L:])
    # an anchor no encode wrote (outside the polygon) is caught, not decoded into symbols
    A[0, 2, 0], A[0, 2, 1] = 3.0, -2.0
    pos = torch.tensor([2 * L, 0, -1, 3 * L, 4 * L], dtype=torch.int64, device="cuda")
    acc = torch.empty(5, dtype=torch.int16, device="cuda")
    fq.fa_access(ctx, A, 1, 3 * L, 3 * L, pos, 5, acc)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == fq.FA_FLAG_CORRUPT | fq.FA_FLAG_RANGE
    h = to_host(acc)
    assert h[0] == 0xFFFF and h[1] == sym[0, 0] and np.all(h[2:] == 0xFFFF)
    ctx.close()


@pytest.mark.parametrize("name", sorted(synth.ARCHIVE_WORKLOADS))
def test_full_size_workload_round_trip_and_sampled_oracle(name):
    """The benchmark's workloads at full size: lossless round trip and random access of every
    sampled position; the oracle recomputes a sample of segments' anchors."""
    w = synth.ARCHIVE_WORKLOADS[name]
    ctx, r, L = make(w.N)
    sym = synth.symbol_streams(w.n_streams, w.T, w.N, w.law)
    A = fq.alloc_archive(ctx, w.n_streams, w.T)
    fq.fa_encode(ctx, to_dev(sym), w.n_streams, w.T, w.T, 0, A)
    out = torch.empty((w.n_streams, w.T), dtype=torch.int16, device="cuda")
    fq.fa_decode(ctx, A, w.n_streams, w.T, w.T, out)
    pos = synth.stream_positions(w.n_streams, w.T, w.T, w.lookups)
    acc = torch.empty(w.lookups, dtype=torch.int16, device="cuda")
    fq.fa_access(ctx, A, w.n_streams, w.T, w.T, torch.from_numpy(pos).cuda(), w.lookups, acc)
    torch.cuda.synchronize()
    assert fq.fa_status(ctx) == 0
    np.testing.assert_array_equal(to_host(out), sym)
    np.testing.assert_array_equal(to_host(acc), sym[pos // w.T, pos % w.T])
    got = A.cpu().numpy()
    S = got.shape[1]
    rng = np.random.default_rng(7)
    V = ofa.vertices(w.N)
    for q, s in zip(rng.integers(0, w.n_streams, 400), rng.integers(0, S, 400)):
        want = ofa.encode_segment(sym[q, s * L:min(s * L + L, w.T)], w.N, r, V=V)
        np.testing.assert_allclose(got[q, s], want, rtol=0, atol=ANCHOR_TOL)
    ctx.close()


def test_access_queue_with_uneven_walks_and_bad_positions():
    """Lookups whose walks differ as much as possible, grouped so that some warps' lanes get only
    zero-step lookups (the anchor's own symbol) and others only full walks, mixed with positions
    outside the batch, repeats, and a count that is not a multiple of a warp's queue."""
    N = 64
    ctx, r, L = make(N)
    nS, T_cap, T = 4, 1000, 997
    sym = synth.symbol_streams(nS, T, N, sub=5)
    A = fq.alloc_archive(ctx, nS, T_cap)
    fq.fa_encode(ctx, to_dev(sym), nS, T, T_cap, 0, A)
    rng = np.random.default_rng(2)
    q = rng.integers(0, nS, size=3000)
    seg = rng.integers(0, T // L, size=3000)
    zero_step = q * T_cap + seg * L + L - 1                    # the anchor's own symbol
    full_walk = q * T_cap + seg * L                             # L - 1 backward steps
    mixed = synth.stream_positions(nS, T_cap, T, 3000, sub=3)
    pos = np.concatenate([zero_step[:1024], full_walk[:1024], mixed, zero_step[1024:], full_walk[1024:2000]])
    bad_at = np.arange(5, len(pos), 7)
    pos[bad_at] = np.where(bad_at % 2, -3, nS * T_cap + 11)
    pos[bad_at[::3]] = T_cap + T                                # position T of stream 1: past the end
    pos = pos[:len(pos) - 13]
    want = np.where(np.isin(np.arange(len(pos)), bad_at), 0xFFFF, 0).astype(np.uint16)
    ok = want == 0
    want[ok] = sym[pos[ok] // T_cap, pos[ok] % T_cap]
    for n in (len(pos), 1, 31, 257):
        acc = torch.empty(n, dtype=torch.int16, device="cuda")
        fq.fa_access(ctx, A, nS, T_cap, T, torch.from_numpy(pos[:n].copy()).cuda(), n, acc)
        torch.cuda.synchronize()
        flags = fq.fa_status(ctx)
        assert flags == (fq.FA_FLAG_RANGE if (~ok[:n]).any() else 0)
        np.testing.assert_array_equal(to_host(acc), want[:n])
    ctx.close()
