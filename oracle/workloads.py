"""The oracle's rotation and codebook for each synthetic workload (TEST INFRASTRUCTURE ONLY).

Combines the seeded draws of ``synth`` with ``oracle.codebook``. Results are cached per process.
Both are shipped to the library as fp32, so the oracle rounds them to fp32 too and every consumer
(oracle and library) sees the same numbers.
"""
from __future__ import annotations

import functools

import numpy as np

import synth
from oracle import codebook as cb


@functools.lru_cache(maxsize=None)
def rotation(cfg: int) -> np.ndarray:
    """fp32 shared rotation of workload ``cfg``."""
    w = synth.WORKLOADS[cfg]
    return cb.haar_rotation(synth.rotation_gaussian(cfg, w.d)).astype(np.float32)


@functools.lru_cache(maxsize=None)
def codebook(cfg: int) -> np.ndarray:
    """fp32 codebook [N, k] of workload ``cfg`` (deterministic init + multi-restart Lloyd)."""
    w = synth.WORKLOADS[cfg]
    Y = cb.source_points(synth.source_gaussians(cfg, w.lloyd_train, w.d), w.k)
    restarts = [synth.restart_gaussian(cfg, w.k, r) for r in range(1, w.lloyd_restarts)]
    C, _ = cb.build_codebook(w.codebook_kind, w.d, w.k, w.N, Y, w.lloyd_iters, restarts,
                             synth.kronecker_offset(cfg))
    return C.astype(np.float32)
