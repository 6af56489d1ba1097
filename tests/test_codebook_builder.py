"""The library's host codebook builder agrees with the oracle's independent one."""
import numpy as np
import pytest

from oracle import codebook as ocb
from oracle import workloads as ow
from random_access_kv_gb300 import codebook as pcb


@pytest.mark.parametrize("cfg", [1, 2])
def test_builder_matches_oracle(cfg):
    C, Pi = pcb.for_workload(cfg)
    np.testing.assert_allclose(Pi, ow.rotation(cfg), atol=1e-7)
    np.testing.assert_allclose(C, ow.codebook(cfg), atol=1e-6)


@pytest.mark.parametrize("d,k,N,kind", [(64, 4, 1024, "kronecker"), (128, 8, 4096, "kronecker"),
                                        (64, 64, 256, "sphere"), (64, 2, 64, "spiral"),
                                        (96, 3, 8, "fibsphere"), (96, 3, 512, "fibsphere")])
def test_initialisation_matches_oracle(d, k, N, kind):
    s = 0.5 if kind != "sphere" else 0.3
    np.testing.assert_allclose(pcb.initial(kind, d, k, N, s), ocb.initial_codebook(kind, d, k, N, s),
                               rtol=1e-7, atol=1e-9)


def test_radii_agree_for_every_k():
    for d, k, N in [(64, 2, 256), (64, 4, 1024), (128, 8, 4096), (64, 1, 16), (96, 3, 512)]:
        np.testing.assert_allclose(pcb.radii(d, k, N), ocb.companded_radii(d, k, N), rtol=1e-10)
