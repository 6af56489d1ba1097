"""Parity checks of the library's outputs against the oracle (test helper).

Tolerances, from the codec's contract and the arithmetic of the fp32/fp16 device path:
  nu       : |nu_gpu - nu| <= 1e-6 nu (fp32 sum of squares of fp16-exact inputs).
  indices  : >= 99.99% of block indices equal the oracle's; every mismatch is a near tie,
             D(c_gpu) - D(c_oracle) <= 1e-5 (|u_b|^2 + |c_oracle|^2), D the fp64 squared
             distance to the oracle's u_b (several indices are correct when distances tie).
  packing  : bit-exact: the oracle's packer applied to the device's indices reproduces the
             device's words (tail bits of the last word zero).
  decode   : device decode of the device's codes within 1e-4 nu (max-abs) of the oracle's fp64
             decode of the same codes, before the fp16 rounding; after it, plus half an fp16 ulp
             of the oracle's value.
  attention: fused attention (fp32 throughout) within, per output element,
               u [ 2 lam (d + sqrt d + 2) A V_inf + lam (2 sqrt(T + 64) + sqrt d + 8) sqrt d V_2 ]
             of the oracle's fp64 attention over the decoded keys and values; u = 2^-24,
             A = scale |q| max_t |k_hat_t| bounds the scores, V_inf / V_2 = max_t of |v_hat_t| in
             the max / Euclidean norm. First term: the score error (rotation of q, d-term dot
             products, the two scalings) moves the softmax output by at most twice the score error
             times V_inf. Second term: the value sums of up to T + 64 terms, the normaliser and
             the d-term inverse rotation. Each sum of n rounded terms is bounded by
             lam sqrt(n) u (Higham and Mary's probabilistic rounding-error bound, lam = 8: it
             fails with probability below 2 exp(-lam^2 / 2) ~ 3e-14 per sum).
"""
from __future__ import annotations

import numpy as np

from oracle import fibquant as ofq

NEAR_TIE_REL = 1e-5
AGREEMENT = 0.9999
DECODE_REL = 1e-4
NU_REL = 1e-6


def fp16_half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - 10)


def check_nu(nu_gpu, nu_orc):
    nu_gpu = np.asarray(nu_gpu, dtype=np.float64)
    err = np.abs(nu_gpu - nu_orc)
    bad = err > NU_REL * nu_orc + 1e-30
    assert not bad.any(), f"nu mismatch at rows {np.flatnonzero(bad)[:5]}: {nu_gpu[bad][:5]} vs {nu_orc[bad][:5]}"


def check_indices(x, C, Pi, idx_gpu, rows=None, agreement=AGREEMENT):
    """Returns (agreement fraction, number of mismatches, max relative gap of mismatches, nu).
    `agreement` is lowered only for inputs built to sit on near ties."""
    C64 = np.asarray(C, dtype=np.float64)
    k = C64.shape[1]
    nu, idx_orc = ofq.encode(x, C, Pi)
    u = ofq.split_blocks(ofq.rotate_normalise(x, Pi, nu), k)
    idx_gpu = np.asarray(idx_gpu, dtype=np.int64)
    assert idx_gpu.shape == idx_orc.shape
    mism = np.argwhere(idx_gpu != idx_orc)
    worst = 0.0
    for m, b in mism:
        ub = u[m, b]
        dg = np.sum((ub - C64[idx_gpu[m, b]]) ** 2)
        do = np.sum((ub - C64[idx_orc[m, b]]) ** 2)
        scale = np.sum(ub * ub) + np.sum(C64[idx_orc[m, b]] ** 2)
        gap = (dg - do) / scale if scale > 0 else np.inf
        worst = max(worst, gap)
        assert gap <= NEAR_TIE_REL, f"row {m} block {b}: index {idx_gpu[m, b]} vs {idx_orc[m, b]}, gap {gap:.3e}"
    agree = 1.0 - len(mism) / max(1, idx_orc.size)
    assert agree >= agreement, f"index agreement {agree:.6f} < {agreement}"
    return agree, len(mism), worst, nu


def check_packing(words_gpu, idx_gpu, B):
    want = ofq.pack(idx_gpu, B)
    got = np.asarray(words_gpu).view(np.uint32)[:want.size]
    np.testing.assert_array_equal(got, want)


def check_decode(out_gpu, nu, idx, C, Pi, fp16_output: bool):
    ref = ofq.decode(nu, idx, C, Pi)
    out = np.asarray(out_gpu, dtype=np.float64)
    tol = DECODE_REL * np.asarray(nu, dtype=np.float64)[:, None]
    if fp16_output:
        tol = tol + fp16_half_ulp(ref)
    err = np.abs(out - ref)
    bad = err > tol
    assert not bad.any(), f"decode error {err[bad][:5]} > tol {tol[bad][:5]} at {np.argwhere(bad)[:3]}"
    nz = np.asarray(nu) > 0
    return float((err[nz] / np.asarray(nu)[nz, None]).max()) if nz.any() else 0.0


ATT_LAMBDA = 8.0


def attention_tolerance(q, K_hat, V_hat, scale) -> np.ndarray:
    """Per-query max-abs tolerance of the fused attention output (see the module docstring)."""
    u = 2.0 ** -24
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    T, d = K_hat.shape
    A = abs(scale) * np.linalg.norm(q, axis=1) * np.linalg.norm(K_hat, axis=1).max()
    v_inf = np.abs(V_hat).max()
    v_2 = np.linalg.norm(V_hat, axis=1).max()
    lam = ATT_LAMBDA
    return u * (2 * lam * (d + np.sqrt(d) + 2) * A * v_inf
                + lam * (2 * np.sqrt(T + 64) + np.sqrt(d) + 8) * np.sqrt(d) * v_2)


def check_attention(out_gpu, q, nu_k, idx_k, nu_v, idx_v, C, Pi, scale):
    """Fused attention of one group's queries vs the oracle. Returns the max of error / tolerance."""
    from oracle import attention as oat
    ref = oat.attention_decode(q, nu_k, idx_k, nu_v, idx_v, C, Pi, scale)
    K_hat = ofq.decode(nu_k, idx_k, C, Pi)
    V_hat = ofq.decode(nu_v, idx_v, C, Pi)
    tol = attention_tolerance(q, K_hat, V_hat, scale)[:, None]
    err = np.abs(np.asarray(out_gpu, dtype=np.float64) - ref)
    bad = err > tol
    assert not bad.any(), f"attention error {err[bad][:5]} > tol {np.broadcast_to(tol, err.shape)[bad][:5]}"
    return float((err / tol).max())
