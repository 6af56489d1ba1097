"""Failure detection without a GPU fault: a bounded device-side wait that nothing completes gives
up and reports FQ_FLAG_TIMEOUT through fq_status, after which the context keeps working; a forced
allocation failure returns FQ_ENOMEM and leaves nothing behind."""
import os
import time

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


def test_bounded_wait_gives_up_and_reports_then_the_context_works():
    C, Pi = ow.codebook(1), ow.rotation(1)
    ctx = fq.fq_codebook_load(C, Pi)
    assert fq.fq_status(ctx) == 0
    t0 = time.perf_counter()
    fq.fq_selftest_wait(ctx, 20_000_000)                     # 20 ms
    flags = fq.fq_status(ctx)
    elapsed = time.perf_counter() - t0
    assert flags == fq.FQ_FLAG_TIMEOUT
    assert 0.015 < elapsed < 5.0
    assert fq.fq_status(ctx) == 0                            # read and cleared
    # the context and the device are still usable: an encode and a decode match the oracle
    x = synth.gaussian_rows(1, 5, 300, 64)
    nu, codes = fq.alloc_store(ctx, 300)
    fq.fq_encode(ctx, torch.from_numpy(x).cuda(), 300, nu, codes)
    out = torch.empty((300, 64), dtype=torch.float32, device="cuda")
    fq.fq_decode_gather_f32(ctx, nu, codes, 300, torch.arange(300, device="cuda"), 300, out)
    torch.cuda.synchronize()
    assert fq.fq_status(ctx) == 0
    idx = ofq.unpack(codes.cpu().numpy().view(np.uint32), 300, 32, 4)
    parity.check_indices(x, C, Pi, idx)
    parity.check_decode(out.cpu().numpy(), nu.cpu().numpy(), idx, C, Pi, fp16_output=False)
    with pytest.raises(fq.FQError):
        fq.fq_selftest_wait(ctx, 2_000_000_000)              # limits above one second are refused
    ctx.close()


def test_forced_allocation_failure_returns_enomem():
    C, Pi = ow.codebook(1), ow.rotation(1)
    os.environ["FQ_TEST_FAIL_ALLOC"] = "1"
    try:
        with pytest.raises(fq.FQError) as e:
            fq.fq_codebook_load(C, Pi)
        assert e.value.code == 2
    finally:
        del os.environ["FQ_TEST_FAIL_ALLOC"]
    ctx = fq.fq_codebook_load(C, Pi)                         # and the next load succeeds
    assert fq.fq_shape(ctx) == (64, 2, 16)
    ctx.close()
