"""fp64 oracle of attention over FibQuant-compressed keys and values (TEST INFRASTRUCTURE ONLY).

[FibQuant §5] stresses that the fixed-address, random-access interface is what allows
decompression to be fused into attention kernels. This states the plain computation such a fused
kernel must reproduce: decode the cached keys and values with the codec's decoder [FibQuant §2.3]
and apply single-query softmax attention,

    o = sum_t p_t v_hat_t / sum_t p_t,   p_t = exp(s_t - max s),   s_t = scale * (q . k_hat_t).

The attention-output cosine [FibQuant §4.2, the fidelity measure of the GPT-2 experiments] compares
o with the same attention over the uncompressed keys and values.
"""
from __future__ import annotations

import numpy as np

from oracle import fibquant as ofq


def softmax_attention(q, K, V, scale) -> np.ndarray:
    """o = softmax(scale * K q) V for one query q [d], keys K [T, d], values V [T, d] (fp64)."""
    s = scale * (np.asarray(K, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    s -= s.max()
    p = np.exp(s)
    p /= p.sum()
    return p @ np.asarray(V, dtype=np.float64)


def attention_decode(q, nu_k, idx_k, nu_v, idx_v, C, Pi, scale) -> np.ndarray:
    """Attention of the queries q [Q, d] of one group over its T decoded keys (norms nu_k [T],
    indices idx_k [T, d/k]) and values (nu_v, idx_v). Returns [Q, d] fp64."""
    K = ofq.decode(nu_k, idx_k, C, Pi)
    V = ofq.decode(nu_v, idx_v, C, Pi)
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    return np.stack([softmax_attention(qr, K, V, scale) for qr in q])


def cosine(a, b) -> np.ndarray:
    """Row-wise cosine similarity, the attention-output fidelity measure of [FibQuant §4.2]."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.sum(a * b, axis=1) / (np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1))
