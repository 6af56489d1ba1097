"""The multi-GPU path is replicas only: every rank runs the workload on its own GPU, with no
collective on the data path; the job's time is its slowest rank's and the job's throughput counts
every rank's units. These CPU tests run two gloo ranks through bench.py's reduction and reporting
logic (the GPU runs use the same functions over NCCL)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, world, local = bench.dist_env()
dist.init_process_group("gloo", rank=rank, world_size=world)
slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)      # rank r took 10 + 5 r ms
value = bench.job_value(1000, 4, world, slowest)
dist.barrier()
print(json.dumps({{"rank": rank, "world": world, "local": local, "slowest": slowest, "value": value}}))
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code: str, world: int, extra=None, timeout=180):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE=str(world), LOCAL_RANK=str(r), **(extra or {}))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=timeout)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    outs = _run_ranks(RANK_SCRIPT.format(root=ROOT), 2)
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs), key=lambda d: d["rank"])
    assert [d["rank"] for d in res] == [0, 1] and all(d["world"] == 2 for d in res)
    assert [d["local"] for d in res] == [0, 1]
    for d in res:
        assert d["slowest"] == 15.0
        assert d["value"] == pytest.approx(2 * 1000 * 4 / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_value(10, 2, 1, 4.0) == pytest.approx(5000.0)


def test_reference_arm_prints_on_rank_zero_only():
    # Under torchrun the other ranks exit 0 without work or output.
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


@pytest.mark.parametrize("mode", [["--archive"], ["--attend", "--workload", "2"], ["--rate-sweep"]])
def test_other_modes_print_on_rank_zero_only(mode):
    # The archive, attention and rate-sweep reference arms follow the same rule.
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *mode,
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
