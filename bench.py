#!/usr/bin/env python3
"""Throughput of the FibQuant codec hot path on one GB300 (or N independent replicas).

One step = the whole hot path over one batch of the Llama-shaped long-context KV workload (the
default; `--workload 1|2|3|5` times the other workloads the same way): 32 layers x 8 KV heads x
32,768 tokens, d = 128, k = 8, N = 4096, b = 1.5 bits per coordinate. K and V arrive as a token
stream: 32 appends, each encoding 1,024 new tokens of every (layer, head) sequence of both
tensors (524,288 vectors per append: norm, rotation, nearest codeword, fixed-address packing),
then a random-access decode of 3,277 token positions (10%) of every sequence (1,677,824 rows:
gather, unpack, codeword lookup, inverse rotation, scaling). K and V share the codebook and live
in one code store, so each append is one launch and the gather one launch. Inputs are resident in
HBM when the timed region starts; L2 is flushed (a 256 MB write) before every timed step, outside
the step's events. The metric is vectors/s (encoded + decoded), with fp16 GB/s beside it. A
step's events bracket all of its launches; the roofline's per-kernel times come from each
kernel's launches timed on their own, L2 flushed before them. `ms_per_step` is the mean of the K
timed steps (their median is reported beside it).

`--attend` times fused decode-into-attention instead: the workload's K and V are encoded into one
store (untimed), then each step is one launch in which one fp16 query per (layer, head) group
attends over all T cached tokens of its group, decoding keys and values inside the kernel. The
metric is then cached K/V vectors read per second, and the line carries the attention-output
cosine against the same attention over the uncompressed fp16 K/V.

`--rate-sweep` measures relative MSE and encode/decode throughput against bits per coordinate,
through the library, for the scalar Lloyd-Max codec (k = 1) and FibQuant at k = 2, 4, 8 and d;
`--sweep-d 96` does it at d = 96 for k = 1, 2, 3 (the Fibonacci-sphere code) and 4.

`--lloyd` times the workload's codebook construction: host numpy Lloyd against GPU Lloyd (the
library's encoder assigns, `fq_centroid_sums` forms the centroids).

`--archive [--archive-workload document|kv-streams]` times the iterated-map archive of symbol
streams (the storage layer of "Fractal KV-Cache Archives"): one step encodes every symbol of the
streams into anchors, decodes them all back and reads a batch of random positions. The metric is
symbols per second through encode and decode; the line also carries each kernel's rate and the
latency of one random access and of one appended symbol, each a single launch.

`--impl reference` times the CPU oracle (the plain fp64 statement of the codec) on a bounded
sample of the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 4]
                    [--attend | --archive [--archive-workload W] | --rate-sweep [--sweep-d 96] | --lloyd]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "KV vectors/s encoded and decoded (fp16 GB/s) per bitrate; % of HBM/TC roofline"
ATTEND_METRIC = "cached KV vectors/s attended (fused decode-into-attention)"
ARCHIVE_METRIC = "archive symbols/s (encode + decode round trip, with a batch of random accesses)"
# fp64 arithmetic instructions the archive kernels issue: a forward or a backward step is a
# subtract and a fused multiply-add per coordinate.
FA_FWD_FP64, FA_BWD_FP64 = 4, 4
# fp64 instructions per SM per clock: the nominal 1.25 TFLOP/s of GB300 over 2 flops per fused
# multiply-add, 152 SMs and the 2070 MHz maximum clock.
FA_FP64_PER_SM_CLK = 2.0
L2_FLUSH_BYTES = 256 << 20


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's); x itself at N = 1."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank_step: int, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank_step * steps / (max_total_ms / 1e3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured",
                "sms": 152}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback", "sms": 152}


# The source file of each timed kernel; its hash (with the shared headers) ties a committed ncu
# traffic figure to the code it measured.
KERNEL_SOURCES = {"encode_k2_tc": ["fq_encode_k2.cu"], "encode_kq_tc": ["fq_encode_kq.cu", "fq_tmem_red.cuh"],
                  "encode_k4_grid": ["fq_encode_k4.cu", "fq_grid4.h"],
                  "encode_full_tc": ["fq_encode_full_tc.cu", "fq_tmem_red.cuh"], "decode_tc": ["fq_decode_tc.cu"],
                  "decode_ws": ["fq_decode_tc.cu"],
                  "decode_full": ["fq_full.cu"], "attend": ["fq_attend_kernel.cuh"],
                  "archive_encode": ["fa_archive.cu"], "archive_decode": ["fa_archive.cu"],
                  "archive_access": ["fa_archive.cu"]}


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "random_access_kv_gb300", "csrc")
    # The kernel's file and the device-code headers it includes (fq_internal.h holds host-side
    # declarations and the context struct, which change without changing any kernel).
    for name in KERNEL_SOURCES[kernel] + ["fq_sm100.cuh", "fq_bits.cuh"]:
        with open(os.path.join(cdir, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def kernel_of(w, op: str) -> str:
    """Name of the kernel that runs `op` ("encode" or "decode") for workload w."""
    if op == "encode":
        if w.k == w.d:
            return "encode_full_tc"
        return {2: "encode_k2_tc", 4: "encode_k4_grid"}.get(w.k, "encode_kq_tc")
    if w.k == w.d:
        return "decode_full"
    return "decode_ws" if w.d == 128 else "decode_tc"


def committed_traffic(kernel: str, workload, rows_per_launch: int):
    """DRAM bytes per launch from profiles/<kernel>_w<workload>.md (profiles/<kernel>_<workload>.md
    for a named workload), if that capture was taken on the kernel's current sources; a capture of
    a smaller case is scaled by rows (traffic grows in proportion to the rows, symbols or lookups a
    launch processes)."""
    stem = f"{kernel}_w{workload}" if isinstance(workload, int) else f"{kernel}_{workload}"
    p = os.path.join(ROOT, "profiles", stem + ".md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().lstrip("- ").startswith(
                    ("source_hash", "dram_bytes_per_launch", "rows_per_launch")):
                k, v = line.split(":", 1)
                vals[k.strip().lstrip("- ")] = v.strip().strip("`")
    if vals.get("source_hash") != source_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"]) * rows_per_launch / float(vals["rows_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_bytes(w, R: int) -> tuple[int, int]:
    """Algorithmic HBM bytes per encoded row and per gathered row."""
    enc = 2 * w.d + 4 + R / 8                # read x fp16, write nu fp32 and the R-bit record
    gat = 8 + 4 + R / 8 + 2 * w.d            # read idx int64, nu, record; write x_hat fp16
    return enc, gat


# ----------------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline leg): the fp64 oracle as it stands.

def oracle_sample_rows(cfg: int) -> tuple[int, int]:
    """Rows per tensor encoded and rows gathered per tensor in one bounded oracle step."""
    return {2: (8192, 4096)}.get(cfg, (2048, 1024))


def time_oracle(cfg: int, steps: int) -> dict:
    from oracle import fibquant as ofq
    from oracle import workloads as ow
    w = synth.WORKLOADS[cfg]
    C, Pi = ow.codebook(cfg), ow.rotation(cfg)
    enc_rows, gat_rows = oracle_sample_rows(cfg)
    xs = [synth.kv_tensor(cfg, t, rows=enc_rows) for t in range(w.tensors)]
    sels = [synth.gather_indices(cfg, t, enc_rows, gat_rows) for t in range(w.tensors)]
    vecs = 0
    t0 = time.perf_counter()
    for _ in range(steps):
        for x, sel in zip(xs, sels):
            nu, idx = ofq.encode(x, C, Pi)
            words = ofq.pack(idx, w.B)
            back = ofq.unpack(words, enc_rows, w.d // w.k, w.B)
            ofq.decode(nu[sel], back[sel], C, Pi).astype(np.float16)
            vecs += enc_rows + gat_rows
    dt = time.perf_counter() - t0
    return {"value": vecs / dt, "seconds": dt, "vectors": vecs,
            "sample": f"{w.tensors} x ({enc_rows} rows encoded + packed, {gat_rows} gathered + decoded) per step "
                      f"of workload {cfg}, {steps} steps, numpy fp64"}


def attend_groups(w) -> tuple[int, int]:
    """(groups, tokens per group) of a two-tensor workload: a group is one (layer, head[, batch])
    sequence of T = shape[-2] tokens, contiguous in the tensor's rows."""
    T = int(w.shape[-2])
    return w.rows // T, T


def time_oracle_attend(cfg: int, steps: int) -> dict:
    from oracle import attention as oat
    from oracle import fibquant as ofq
    from oracle import workloads as ow
    w = synth.WORKLOADS[cfg]
    C, Pi = ow.codebook(cfg), ow.rotation(cfg)
    _, T = attend_groups(w)
    groups = 2
    x = [synth.kv_tensor(cfg, t, rows=groups * T) for t in range(2)]
    q = synth.query_rows(cfg, groups, w.d)
    t0 = time.perf_counter()
    for _ in range(steps):
        enc = [ofq.encode(xt, C, Pi) for xt in x]
        for g in range(groups):
            sl = slice(g * T, (g + 1) * T)
            oat.attention_decode(q[g], enc[0][0][sl], enc[0][1][sl], enc[1][0][sl], enc[1][1][sl], C, Pi,
                                 1.0 / np.sqrt(w.d))
    dt = time.perf_counter() - t0
    vecs = steps * groups * 2 * T
    return {"value": vecs / dt, "seconds": dt, "vectors": vecs,
            "sample": f"{groups} groups x {T} tokens of workload {cfg} (K and V encoded, then decoded and "
                      f"attended by one query each), {steps} steps, numpy fp64"}


def archive_params(N: int) -> tuple[float, int]:
    """(r, L) of the archive benchmark: r = 3/4 of the disjointness limit sin(pi/N) / (1 + sin(pi/N)),
    L the longest segment the fp64 error bound allows (the library's own bound)."""
    import random_access_kv_gb300 as fq
    r = 0.75 * fq.fa_ratio_limit(N)
    return r, fq.fa_max_segment(N, r)


ARCHIVE_ORACLE_SYMBOLS = 300000


def time_oracle_archive(name: str, steps: int) -> dict:
    """The oracle's encode, backward-search decode and random access on a bounded sample: the first
    streams of the workload (their first symbols for a single long stream), about 300,000 symbols
    per step, and one random position read back per 16 symbols."""
    from oracle import fractal as ofa
    w = synth.ARCHIVE_WORKLOADS[name]
    r = 0.75 * ofa.ratio_limit(w.N)
    L = ofa.max_segment(w.N, r)
    ns = min(w.n_streams, -(-ARCHIVE_ORACLE_SYMBOLS // w.T))
    T = min(w.T, ARCHIVE_ORACLE_SYMBOLS)
    sym = synth.symbol_streams(w.n_streams, w.T, w.N, w.law)[:ns, :T]
    pos = synth.stream_positions(ns, T, T, ns * T // 16)
    t0 = time.perf_counter()
    for _ in range(steps):
        A = ofa.encode(sym, w.N, r, L)
        ofa.decode(A, T, w.N, r, L)
        for p in pos:
            ofa.access(A, T, w.N, r, L, int(p) // T, int(p) % T)
    dt = time.perf_counter() - t0
    return {"value": steps * ns * T / dt, "seconds": dt, "symbols": steps * ns * T,
            "sample": f"{ns} stream(s) x {T} symbols of workload '{name}' (encoded, decoded, and "
                      f"{ns * T // 16} random positions read back), {steps} steps, Python fp64"}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.archive:
        def timer(_, n):
            return time_oracle_archive(args.archive_workload, n)
        name, metric, unit = synth.ARCHIVE_WORKLOADS[args.archive_workload].name, ARCHIVE_METRIC, "symbols/s"
    else:
        timer = time_oracle_attend if args.attend else time_oracle
        name, metric, unit = synth.WORKLOADS[args.workload].name, ATTEND_METRIC if args.attend else METRIC, "vectors/s"
    timer(args.workload, max(1, args.warmup))
    r = timer(args.workload, args.steps)
    cores = 1 if args.archive else host_cores()        # the archive oracle is plain Python
    line = {
        "impl": "reference", "metric": metric, "value": r["value"], "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * r["seconds"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "sample": r["sample"]},
        "cpu_baseline": {"value": r["value"], "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# GPU arm.

def run_ours(args) -> None:
    import torch
    import random_access_kv_gb300 as fq
    from random_access_kv_gb300 import build as fbuild
    from random_access_kv_gb300 import codebook as pcb

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    if world > 1:
        torch.distributed.barrier()

    cfg = args.workload
    w = synth.WORKLOADS[cfg]
    if w.op not in ("encode+gather", "encode+decode", "stream+gather"):
        raise SystemExit(f"workload {cfg} ({w.op}) is not timed by bench.py")
    streaming = w.op == "stream+gather"
    if streaming and args.rows and args.rows % w.shape[-2]:
        raise SystemExit(f"--rows must be a multiple of the sequence length {w.shape[-2]} here")
    gathers = w.op != "encode+decode"            # encode+decode workloads decode every row
    C, Pi = pcb.for_workload(cfg)
    ctx = fq.fq_codebook_load(C, Pi, local)
    R = fq.fq_record_bits(ctx)
    M, d, nt = (w.rows if not args.rows else min(args.rows, w.rows)), w.d, w.tensors
    # K and V share the codebook and rotation, so they share one code store: rows [t*M, (t+1)*M)
    # hold tensor t. One encode launch covers all tensors, one decode launch all decoded rows.
    MT = nt * M
    if streaming:
        # (layer, head) sequences of capacity T per tensor; each append adds `new` tokens to all.
        n_seq, T, new = M // w.shape[-2], w.shape[-2], w.stream_new
        n_steps = T // new
        pos = synth.token_positions(cfg, T, w.gather)
        per = (np.arange(n_seq)[:, None] * T + pos[None, :]).reshape(-1)
        idx_np = np.concatenate([t * M + per for t in range(nt)]).astype(np.int64)

        def arrival_order(a):  # [n_seq*T, d] -> [steps, n_seq, new, d], the order tokens arrive in
            return np.ascontiguousarray(a.reshape(n_seq, n_steps, new, d).transpose(1, 0, 2, 3))
        x_np = np.concatenate([arrival_order(synth.kv_tensor(cfg, t, rows=M if M < w.rows else None))
                               for t in range(nt)], axis=1)
        x_np = x_np.reshape(n_steps, nt * n_seq * new, d)
    else:
        x_np = np.concatenate([synth.kv_tensor(cfg, t, rows=M) for t in range(nt)])
        if gathers:
            idx_np = np.concatenate([t * M + synth.gather_indices(cfg, t, M, min(w.gather, M)) for t in range(nt)])
        else:
            idx_np = np.arange(MT, dtype=np.int64)
    G = int(idx_np.size)
    x_host = torch.from_numpy(x_np).pin_memory()
    i_host = torch.from_numpy(idx_np).pin_memory()
    del x_np, idx_np                      # the pinned copies are the inputs from here on
    xs = x_host.to(dev)
    idx = i_host.to(dev)
    nu, codes = fq.alloc_store(ctx, MT, dev)
    out = torch.empty((G, d), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    enc_launches = n_steps if streaming else 1
    launches_per_step = enc_launches + 1

    def encode_all():
        if streaming:
            for st in range(n_steps):
                fq.fq_encode_append(ctx, xs[st], nt * n_seq, new, T, st * new, nu, codes, sp)
        else:
            fq.fq_encode(ctx, xs, MT, nu, codes, 0, sp)

    def decode_all():
        if gathers:
            fq.fq_decode_gather(ctx, nu, codes, MT, idx, G, out, sp)
        else:
            fq.fq_decode(ctx, nu, codes, MT, out, sp)

    def step(ev=None):
        # No event between the launches: each kernel lets the next one be scheduled before it
        # ends (programmatic dependent launch), and an event in between would serialise them.
        if ev is not None:
            ev[0].record(stream)
        encode_all()
        decode_all()
        if ev is not None:
            ev[1].record(stream)

    def timed_alone(fn, reps):
        """Per-kernel device time: fn bracketed by its own events, L2 flushed before each."""
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(a.elapsed_time(b))
        return ms

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fq.fq_status(ctx, sp) != 0:
        raise SystemExit("device flags set during warm-up")

    evs = []
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    for _ in range(args.steps):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        step(ev)
        evs.append(ev)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = sum(step_ms)
    # Per-kernel times for the roofline, each launch timed on its own.
    enc_step_ms = timed_alone(encode_all, max(3, args.steps))
    dec_step_ms = timed_alone(decode_all, max(3, args.steps))
    total_ms = max_over_ranks(total_ms, world, dev)
    flags = fq.fq_status(ctx, sp)

    vec_per_step = MT + G
    value = job_value(vec_per_step, args.steps, world, total_ms)

    # End to end through the public API from pinned host memory, every step: H2D of the inputs,
    # encode, decode, D2H of the norms, codes and decoded rows. The step is cut into row chunks on
    # three streams (copy in, compute, copy out), so that the copies overlap the kernels and each
    # other; the events bracket all of it. Chunks start on whole 32-bit code words (1024-row
    # multiples), so each chunk's records are its own words and a chunk is a store of its own.
    # (Cutting a gathering workload by tensor, so that one tensor's gather and copy-back overlap the
    # next tensor's upload, measured the same on w2: the step moves 66 MB over the host link either
    # way.)
    nu_host = torch.empty_like(nu, device="cpu").pin_memory()
    code_host = torch.empty_like(codes, device="cpu").pin_memory()
    out_host = torch.empty_like(out, device="cpu").pin_memory()
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    if streaming:
        bounds = None
    else:
        # At least 16 MB of input per chunk: each chunk costs tens of microseconds of host-side
        # issue (copies, events, a launch), which smaller chunks would not hide.
        nch = max(1, min(8, (MT * d * 2) // (16 << 20)))
        bounds = sorted({min(MT, (MT * c // nch) // 1024 * 1024) for c in range(nch)} | {MT})

    def words(r):                                   # first code word of row r (r on a word boundary)
        return (r * R + 31) // 32

    def e2e_serial():
        xs.copy_(x_host, non_blocking=True)
        if gathers:
            idx.copy_(i_host, non_blocking=True)
        step()
        nu_host.copy_(nu, non_blocking=True)
        code_host.copy_(codes, non_blocking=True)
        out_host.copy_(out, non_blocking=True)

    def e2e_step():
        if not streaming and len(bounds) == 2:    # one chunk: nothing to overlap
            e2e_serial()
            return
        ev0 = torch.cuda.Event()
        ev0.record(stream)
        for st in (s_in, s_cmp, s_out):
            st.wait_event(ev0)
        if gathers:
            with torch.cuda.stream(s_in):
                idx.copy_(i_host, non_blocking=True)
        if streaming:
            for st in range(n_steps):
                with torch.cuda.stream(s_in):
                    xs[st].copy_(x_host[st], non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
                s_cmp.wait_event(e_in)
                fq.fq_encode_append(ctx, xs[st], nt * n_seq, new, T, st * new, nu, codes, s_cmp.cuda_stream)
        else:
            for a, b in zip(bounds[:-1], bounds[1:]):
                with torch.cuda.stream(s_in):
                    xs[a:b].copy_(x_host[a:b], non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
                s_cmp.wait_event(e_in)
                fq.fq_encode(ctx, xs[a:b], b - a, nu[a:], codes[words(a):], 0, s_cmp.cuda_stream)
                if not gathers:
                    fq.fq_decode(ctx, nu[a:], codes[words(a):], b - a, out[a:b], s_cmp.cuda_stream)
                e_c = torch.cuda.Event()
                e_c.record(s_cmp)
                s_out.wait_event(e_c)
                with torch.cuda.stream(s_out):
                    nu_host[a:b].copy_(nu[a:b], non_blocking=True)
                    code_host[words(a):words(b)].copy_(codes[words(a):words(b)], non_blocking=True)
                    if not gathers:
                        out_host[a:b].copy_(out[a:b], non_blocking=True)
        if gathers:
            e_idx = torch.cuda.Event()                # the index copy and every x chunk have landed
            e_idx.record(s_in)
            s_cmp.wait_event(e_idx)
            fq.fq_decode_gather(ctx, nu, codes, MT, idx, G, out, s_cmp.cuda_stream)
            e_c = torch.cuda.Event()
            e_c.record(s_cmp)
            s_out.wait_event(e_c)
            with torch.cuda.stream(s_out):
                if streaming:
                    nu_host.copy_(nu, non_blocking=True)
                    code_host.copy_(codes, non_blocking=True)
                out_host.copy_(out, non_blocking=True)
        e_end = torch.cuda.Event()
        e_end.record(s_out)
        stream.wait_event(e_end)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    # The pipelined step must hand back what the device-resident step computes.
    got = (out_host.clone(), code_host.clone(), nu_host.clone())
    step()
    torch.cuda.synchronize(dev)
    if not (torch.equal(got[0], out.cpu()) and torch.equal(got[1], codes.cpu()) and torch.equal(got[2], nu.cpu())):
        raise SystemExit("the end-to-end pipeline returned other results than the device-resident step")
    del got
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    h2d = x_host.numel() * 2 + (i_host.numel() * 8 if gathers else 0)
    d2h = nu_host.numel() * 4 + code_host.numel() * 4 + out_host.numel() * 2
    e2e_total = sum(e2e_ms)
    e2e_total = max_over_ranks(e2e_total, world, dev)
    e2e_value = job_value(vec_per_step, args.steps, world, e2e_total)

    enc_b, gat_b = workload_bytes(w, R)
    if not gathers:
        gat_b -= 8                          # a full decode reads no index array
    # per launch: a streamed encode is n_steps append launches of MT / n_steps rows each
    enc_ms = statistics.mean(enc_step_ms) / enc_launches
    enc_rows = MT // enc_launches
    gat_ms = statistics.mean(dec_step_ms)
    peaks = measured_peaks()
    dec_name = "decode_gather" if gathers else "decode"
    if enc_ms * enc_launches >= gat_ms:
        dom, dom_bytes, dom_ms, dom_rows = "encode", enc_b * enc_rows, enc_ms, enc_rows
        kname = kernel_of(w, "encode")
    else:
        dom, dom_bytes, dom_ms, dom_rows = dec_name, gat_b * G, gat_ms, G
        kname = kernel_of(w, "decode")
    roofline = {"kernel": dom, "cuda_kernel": kname, "traffic": committed_traffic(kname, cfg, dom_rows),
                "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": int(dom_bytes), "launch_ms": round(dom_ms, 5),
                "encode_launch_ms": round(enc_ms, 5), "encode_rows_per_launch": enc_rows,
                f"{dec_name}_launch_ms": round(gat_ms, 5), f"{dec_name}_rows_per_launch": G,
                "encode_gbs": round(enc_b * enc_rows / (enc_ms / 1e3) / 1e9, 1),
                f"{dec_name}_gbs": round(gat_b * G / (gat_ms / 1e3) / 1e9, 1)}
    if dom == "encode" and kname in ("encode_full_tc", "encode_kq_tc"):
        # An exhaustive nearest-codeword search is a contraction of every block with every
        # codeword, 2 N k flops per block and 2 N d per vector (the full-vector code's, with the
        # rotated codebook). Its time at the tensor pipe's peak is far above the vector's HBM time,
        # so the tensor pipe is the binding roofline; the HBM rate stays beside it (encode_gbs).
        flops = 2.0 * enc_rows * w.N * d
        achieved = flops / (dom_ms / 1e3) / 1e12
        roofline.update({"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "algorithmic_flops_per_launch": flops,
                         "hbm_frac": round(enc_b * enc_rows / (enc_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)})
    else:
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        roofline.update({"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)})
    if w.k < w.d:
        # The other bound of a k <= 8 encode: an exhaustive nearest-codeword search on the CUDA
        # cores, (d/k) N (k + 2) lane instructions per row, against 128 lane instructions per
        # cycle per SM at the sampled clock. Above 1.0 means the search beats exhaustive scanning.
        instr = (d // w.k) * w.N * (w.k + 2)
        sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
        alu_peak = peaks["sms"] * 128 * sm_mhz * 1e6
        enc_rows_s = enc_rows / (enc_ms / 1e3)
        roofline["search_alu"] = {"bound": "alu", "instr_per_row": instr,
                                  "achieved": round(enc_rows_s * instr / 1e12, 2),
                                  "peak": round(alu_peak / 1e12, 2), "unit": "T lane-instr/s",
                                  "frac": round(enc_rows_s * instr / alu_peak, 3)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle(cfg, args.cpu_steps)
        cpu = {"value": r["value"], "unit": "vectors/s", "cores": host_cores(), "kind": "oracle",
               "sample": r["sample"], "seconds": round(r["seconds"], 2)}

    if rank == 0:
        conf = {"workload": w.name + (f" (first {M} rows per tensor)" if M != w.rows else ""), "rows_per_tensor": M, "tensors": nt, "d": d, "k": w.k, "N": w.N,
                "bits_per_coordinate": w.B / w.k, "record_bits": R,
                ("gathered_rows" if gathers else "decoded_rows"): G,
                "layout": "K and V in one code store; one encode and one decode launch per step"
                          + (" (one append launch per token block)" if streaming else ""),
                "l2": "flushed before every timed step (256 MB write, outside the step events)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
        if streaming:
            conf.update({"append_steps": n_steps, "tokens_per_append": new, "sequences": nt * n_seq})
        line = {
            "metric": METRIC, "value": value, "unit": "vectors/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": conf,
            "step_statistic": "mean over the timed steps (ms_per_step); median beside it",
            "median_ms_per_step": statistics.median(step_ms),
            "fp16_gbps": value * 2 * d / 1e9,
            "roofline": roofline,
            "cpu_baseline": cpu,
            # The mean is the value; the spread shows how much of it the shared host link costs.
            "e2e": {"value": e2e_value, "unit": "vectors/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_total / args.steps,
                    "median_ms_per_step": statistics.median(e2e_ms), "min_ms_per_step": min(e2e_ms)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "device_flags": flags,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_attend(args) -> None:
    import torch
    import random_access_kv_gb300 as fq
    from random_access_kv_gb300 import build as fbuild
    from random_access_kv_gb300 import codebook as pcb

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    if world > 1:
        torch.distributed.barrier()

    cfg = args.workload
    w = synth.WORKLOADS[cfg]
    if w.tensors != 2:
        raise SystemExit(f"workload {cfg} has no separate keys and values")
    C, Pi = pcb.for_workload(cfg)
    ctx = fq.fq_codebook_load(C, Pi, local)
    R = fq.fq_record_bits(ctx)
    groups, T = attend_groups(w)
    if args.groups:
        groups = min(groups, args.groups)
    M, d = groups * T, w.d
    qpg = args.q_per_group
    nq = groups * qpg
    scale = 1.0 / float(np.sqrt(d))
    # The cache: K rows [0, M), V rows [M, 2M) of one store, encoded once (untimed).
    nu, codes = fq.alloc_store(ctx, 2 * M, dev)
    for t in range(2):
        x = torch.from_numpy(synth.kv_tensor(cfg, t, rows=M)).to(dev)
        fq.fq_encode(ctx, x, M, nu, codes, t * M)
        del x
    torch.cuda.synchronize(dev)
    q_host = torch.from_numpy(synth.query_rows(cfg, nq, d)).pin_memory()
    q = q_host.to(dev)
    out = torch.empty((nq, d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step():
        fq.fq_attend(ctx, nu, codes, 2 * M, q, nq, qpg, T, 0, M, T, scale, out, sp)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fq.fq_status(ctx, sp) != 0:
        raise SystemExit("device flags set during warm-up")

    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    evs = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(ms)
    total_ms = max_over_ranks(total_ms, world, dev)
    vec_per_step = 2 * groups * T
    value = job_value(vec_per_step, args.steps, world, total_ms)

    # End to end: the cache stays resident (it is the KV cache); each step copies its queries in
    # from pinned host memory and the attention outputs back.
    out_host = torch.empty_like(out, device="cpu").pin_memory()
    e2e_ms = []
    for i in range(args.steps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q.copy_(q_host, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    e2e_total = sum(e2e_ms)
    e2e_total = max_over_ranks(e2e_total, world, dev)
    e2e_value = job_value(vec_per_step, args.steps, world, e2e_total)

    # Fidelity: cosine with exact attention (fp64 on the device) over the uncompressed fp16 K and V,
    # and, as a full-size consistency check of the fused kernel, over the same cache decoded by
    # the library's separate decoder.
    o_fused = out.double()
    cos, cos_dec = [], []
    k_all, v_all = synth.kv_tensor(cfg, 0, rows=M), synth.kv_tensor(cfg, 1, rows=M)

    def attention(Kx, Vx, qx):             # qx [groups, qpg, d]
        p = torch.softmax(scale * torch.einsum("gtd,gqd->gqt", Kx, qx), dim=2)
        return torch.einsum("gqt,gtd->gqd", p, Vx).reshape(-1, d)

    for g0 in range(0, groups, 64):
        g1 = min(groups, g0 + 64)
        n = (g1 - g0) * T
        Kx = torch.from_numpy(k_all[g0 * T:g1 * T]).to(dev).double().view(g1 - g0, T, d)
        Vx = torch.from_numpy(v_all[g0 * T:g1 * T]).to(dev).double().view(g1 - g0, T, d)
        qg = q[g0 * qpg:g1 * qpg].double().view(g1 - g0, qpg, d)
        og = o_fused[g0 * qpg:g1 * qpg]
        cos.append(torch.nn.functional.cosine_similarity(attention(Kx, Vx, qg), og, dim=1).cpu())
        del Kx, Vx
        rows = torch.arange(g0 * T, g1 * T, device=dev)
        dec = torch.empty((2 * n, d), dtype=torch.float32, device=dev)
        fq.fq_decode_gather_f32(ctx, nu, codes, 2 * M, torch.cat([rows, rows + M]), 2 * n, dec, sp)
        dec = dec.double().view(2, g1 - g0, T, d)
        cos_dec.append(torch.nn.functional.cosine_similarity(attention(dec[0], dec[1], qg), og, dim=1).cpu())
        del dec
    del k_all, v_all
    cos = torch.cat(cos).numpy()
    cos_dec = torch.cat(cos_dec).numpy()
    flags = fq.fq_status(ctx, sp)

    launch_ms = statistics.mean(ms)
    alg_bytes = groups * T * 2 * (R / 8 + 4) + nq * d * (2 + 4)
    peaks = measured_peaks()
    achieved = alg_bytes / (launch_ms / 1e3) / 1e9
    roofline = {"kernel": "attend", "cuda_kernel": "attend", "traffic": committed_traffic("attend", cfg, groups * T),
                "peak_source": peaks["source"], "algorithmic_bytes_per_launch": int(alg_bytes),
                "launch_ms": round(launch_ms, 5), "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle_attend(cfg, args.cpu_steps)
        cpu = {"value": r["value"], "unit": "vectors/s", "cores": host_cores(), "kind": "oracle",
               "sample": r["sample"], "seconds": round(r["seconds"], 2)}
    if rank == 0:
        line = {
            "metric": ATTEND_METRIC, "value": value, "unit": "vectors/s", "n_gpus": world, "steps": args.steps,
            "query_token_pairs_per_s": world * nq * T * args.steps / (total_ms / 1e3),
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name + " -- fused attention"
                       + (f" (first {groups} groups)" if groups * T != w.rows else ""), "groups": groups, "tokens_per_group": T,
                       "queries_per_group": qpg, "d": d, "k": w.k, "N": w.N, "record_bits": R,
                       "layout": "K rows [0, M), V rows [M, 2M) of one code store; one launch per step",
                       "l2": "flushed before every timed step (256 MB write, outside the step events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "fidelity": {"attention_cosine_mean": float(cos.mean()), "attention_cosine_min": float(cos.min()),
                         "against": "softmax attention over the uncompressed fp16 K/V, fp64",
                         "queries": "N(0, 1) fp16, independent of the keys",
                         "unfused_cosine_min": float(cos_dec.min()),
                         "unfused": "softmax attention, fp64, over the same cache decoded by fq_decode_gather_f32"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "vectors/s", "h2d_bytes_per_step": int(q_host.numel() * 2),
                    "d2h_bytes_per_step": int(out_host.numel() * 4)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "device_flags": flags,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_archive(args) -> None:
    import torch
    import random_access_kv_gb300 as fq
    from random_access_kv_gb300 import build as fbuild

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    if world > 1:
        torch.distributed.barrier()

    w = synth.ARCHIVE_WORKLOADS[args.archive_workload]
    r, L = archive_params(w.N)
    ctx = fq.fa_create(w.N, r, L, local)
    nS, T = w.n_streams, w.T
    S = fq.fa_segments(ctx, T)
    sym_np = synth.symbol_streams(nS, T, w.N, w.law)
    pos_np = synth.stream_positions(nS, T, T, w.lookups)
    sym_host = torch.from_numpy(sym_np.view(np.int16)).pin_memory()
    pos_host = torch.from_numpy(pos_np).pin_memory()
    sym = sym_host.to(dev)
    pos = pos_host.to(dev)
    A = fq.alloc_archive(ctx, nS, T, dev)
    dec = torch.empty((nS, T), dtype=torch.int16, device=dev)
    acc = torch.empty(w.lookups, dtype=torch.int16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def enc():
        fq.fa_encode(ctx, sym, nS, T, T, 0, A, sp)

    def dcd():
        fq.fa_decode(ctx, A, nS, T, T, dec, sp)

    def rnd():
        fq.fa_access(ctx, A, nS, T, T, pos, w.lookups, acc, sp)

    def step():
        enc()
        dcd()
        rnd()

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fq.fa_status(ctx, sp) != 0:
        raise SystemExit("device flags set during warm-up")
    if not (torch.equal(dec.cpu(), sym_host) and np.array_equal(acc.cpu().numpy(), sym_np[pos_np // T, pos_np % T].view(np.int16))):
        raise SystemExit("the archive did not return the symbols it stored")

    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    evs = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world, dev)
    value = job_value(nS * T, args.steps, world, total_ms)

    def timed_alone(fn, reps):
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.mean(ms)

    reps = max(5, args.steps)
    enc_ms, dec_ms, acc_ms = timed_alone(enc, reps), timed_alone(dcd, reps), timed_alone(rnd, reps)

    # Single-launch latencies, the GPU counterpart of a per-character or per-lookup time: one random
    # access of one position, and one append of one symbol to each stream (an archive with room).
    one = pos[:1].clone()
    lat_acc = timed_alone(lambda: fq.fa_access(ctx, A, nS, T, T, one, 1, acc, sp), 50)
    extra = 40 + 10 * w.append
    cap = T + extra
    A2 = fq.alloc_archive(ctx, nS, cap, dev)
    fq.fa_encode(ctx, sym, nS, T, cap, 0, A2, sp)
    tail = torch.from_numpy(synth.symbol_streams(nS, extra, w.N, w.law, sub=1).view(np.int16)).to(dev)
    cols = [tail[:, i:i + 1].contiguous() for i in range(40)]
    toks = [tail[:, 40 + i * w.append:40 + (i + 1) * w.append].contiguous() for i in range(10)]
    done = [T]

    def append(chunk, n):
        fq.fa_encode(ctx, chunk, nS, n, cap, done[0], A2, sp)
        done[0] += n

    lat_app = timed_alone(lambda: append(cols[done[0] - T], 1), 40)
    lat_tok = timed_alone(lambda: append(toks[(done[0] - T - 40) // w.append], w.append), 10)
    torch.cuda.synchronize(dev)
    full = torch.cat([sym, tail], dim=1).contiguous()
    A3 = fq.alloc_archive(ctx, nS, cap, dev)
    fq.fa_encode(ctx, full, nS, cap, cap, 0, A3, sp)
    if not torch.equal(A2, A3):
        raise SystemExit("appended anchors differ from a one-call encode")

    # End to end: the streams come from pinned host memory, the anchors, the decoded streams and the
    # random-access results go back. (Cutting a batch of streams into four groups on three CUDA
    # streams, so that one group's copies overlap another's kernels, measured slower on kv-streams:
    # 9.4e9 against 1.3e10 symbols/s.)
    a_host = torch.empty_like(A, device="cpu").pin_memory()
    d_host = torch.empty_like(dec, device="cpu").pin_memory()
    r_host = torch.empty_like(acc, device="cpu").pin_memory()
    torch.cuda.synchronize(dev)
    a_ref = A.cpu()                                 # the device-resident step's anchors
    r_ref = torch.from_numpy(np.ascontiguousarray(sym_np[pos_np // T, pos_np % T]).view(np.int16))

    def e2e_step():
        sym.copy_(sym_host, non_blocking=True)
        pos.copy_(pos_host, non_blocking=True)
        step()
        a_host.copy_(A, non_blocking=True)
        d_host.copy_(dec, non_blocking=True)
        r_host.copy_(acc, non_blocking=True)

    e2e_ms = []
    for i in range(args.steps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
        if i == 2:
            # the end-to-end step hands back what the device-resident step computes
            if not (torch.equal(d_host, sym_host) and torch.equal(r_host, r_ref) and torch.equal(a_host, a_ref)):
                raise SystemExit("the end-to-end archive step returned other results than the device step")
    e2e_total = max_over_ranks(sum(e2e_ms), world, dev)
    e2e_value = job_value(nS * T, args.steps, world, e2e_total)
    flags = fq.fa_status(ctx, sp)

    # Roofline: the kernels are chains of dependent fp64 steps, bound by the fp64 pipe.
    seg_len = np.minimum(L, T - np.arange(S) * L)
    t_in = pos_np % T
    acc_steps = int(np.sum(np.minimum(L, T - (t_in // L) * L) - 1 - t_in % L))
    fp64 = {"encode": FA_FWD_FP64 * nS * T, "decode": FA_BWD_FP64 * nS * int(np.sum(seg_len - 1)),
            "access": FA_BWD_FP64 * acc_steps}
    times = {"encode": enc_ms, "decode": dec_ms, "access": acc_ms}
    dom = max(times, key=times.get)
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    peaks = measured_peaks()
    peak = peaks["sms"] * FA_FP64_PER_SM_CLK * sm_mhz * 1e6 / 1e12     # T fp64 instructions / s
    ach = {k: fp64[k] / (times[k] / 1e3) / 1e12 for k in times}
    # The committed capture is of the kv-streams workload; another workload's anchor table differs in
    # size, so its traffic is not a scaled copy of that capture.
    units = {"encode": nS * T, "decode": nS * T, "access": w.lookups}
    traffic = (committed_traffic("archive_" + dom, "kv-streams", units[dom])
               if args.archive_workload == "kv-streams" else None)
    roofline = {"kernel": dom, "cuda_kernel": "archive_" + dom, "traffic": traffic, "bound": "alu",
                "achieved": round(ach[dom], 4), "peak": round(peak, 4), "unit": "T fp64 instr/s",
                "frac": round(ach[dom] / peak, 4), "peak_source": "nominal fp64 rate (2 per SM per clock) at the "
                "sampled SM clock", "fp64_instr_per_launch": fp64[dom], "launch_ms": round(times[dom], 5),
                "per_kernel": {k: {"ms": round(times[k], 5), "fp64_instr": fp64[k], "frac": round(ach[k] / peak, 4)}
                               for k in times}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c = time_oracle_archive(args.archive_workload, args.cpu_steps)
        cpu = {"value": c["value"], "unit": "symbols/s", "cores": 1, "kind": "oracle", "sample": c["sample"],
               "seconds": round(c["seconds"], 2)}
    if rank == 0:
        line = {
            "metric": ARCHIVE_METRIC, "value": value, "unit": "symbols/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "n_streams": nS, "T": T, "N": w.N, "r": r, "L": L,
                       "lookups_per_step": w.lookups, "anchor_bits_per_symbol": round(128 / L, 3),
                       "raw_bits_per_symbol": float(np.log2(w.N)),
                       "l2": "flushed before every timed step (256 MB write, outside the step events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "rates": {"encode_symbols_per_s": nS * T / (enc_ms / 1e3), "decode_symbols_per_s": nS * T / (dec_ms / 1e3),
                      "access_lookups_per_s": w.lookups / (acc_ms / 1e3),
                      "encode_ns_per_symbol": 1e6 * enc_ms / (nS * T),
                      "access_us_single_lookup": 1e3 * lat_acc,
                      "append_us_one_symbol_per_stream": 1e3 * lat_app,
                      "append_us_one_token": 1e3 * lat_tok, "token_symbols_per_stream": w.append},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "symbols/s",
                    "h2d_bytes_per_step": int(sym_host.numel() * 2 + pos_host.numel() * 8),
                    "d2h_bytes_per_step": int(a_host.numel() * 8 + d_host.numel() * 2 + r_host.numel() * 2)},
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
            "device_flags": flags,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        torch.distributed.destroy_process_group()


# Rate sweep: (codec, k, N) points at d = 64; b = log2(N) / k bits per coordinate.
SWEEP_POINTS = ([("scalar", 1, n) for n in (2, 4, 8, 16)]
                + [("fibquant", 2, n) for n in (4, 8, 16, 32, 64, 128, 256)]
                + [("fibquant", 4, n) for n in (16, 64, 256, 1024, 4096)]
                + [("fibquant", 8, n) for n in (256, 4096)]
                + [("fibquant", 64, n) for n in (256, 1024, 4096)])
# d = 96 (a head dimension that 3 divides): integer rates 1, 2, 3 for k = 1, 2, 3 (Fibonacci sphere), 4.
SWEEP_POINTS_96 = ([("scalar", 1, n) for n in (2, 4, 8)]
                   + [("fibquant", 2, n) for n in (4, 16, 64)]
                   + [("fibquant", 3, n) for n in (8, 64, 512)]
                   + [("fibquant", 4, n) for n in (16, 256, 4096)])


def run_rate_sweep(args) -> None:
    """Relative MSE and kernel throughput against bits per coordinate, through the library, for the
    scalar Lloyd-Max codec (k = 1, integer rates only) and FibQuant at k = 2, 4, 8 and d."""
    import torch
    import random_access_kv_gb300 as fq
    from random_access_kv_gb300 import build as fbuild
    from random_access_kv_gb300 import codebook as pcb

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fbuild.build()
    d, rows, seed = args.sweep_d, args.rows or 262144, 1
    sweep = SWEEP_POINTS if d == 64 else SWEEP_POINTS_96
    Pi = pcb.haar(synth.rotation_gaussian(seed, d)).astype(np.float32)
    x_np = synth.gaussian_rows(seed, 3, rows, d)
    x = torch.from_numpy(x_np).to(dev)
    x64 = x.double()
    xx = (x64 * x64).sum(dim=1)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    points = []
    for i, (codec, k, N) in enumerate(sweep):
        t0 = time.perf_counter()
        if codec == "scalar":
            C, _ = pcb.scalar_lloyd_max(d, N)
        else:
            kind = "sphere" if k == d else {2: "spiral", 3: "fibsphere"}.get(k, "kronecker")
            T = int(min(131072, max(32768, 32 * N)))
            C, _ = pcb.build(kind, d, k, N, synth.source_gaussians(seed, T, d, chunk=100 + i), 10)
        build_s = time.perf_counter() - t0
        ctx = fq.fq_codebook_load(C.astype(np.float32), Pi, local)
        nu, codes = fq.alloc_store(ctx, rows, dev)
        out = torch.empty((rows, d), dtype=torch.float16, device=dev)
        enc_ms, dec_ms = [], []
        for rep in range(3 + args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            flush.zero_()
            ev[0].record(stream)
            fq.fq_encode(ctx, x, rows, nu, codes, 0, sp)
            ev[1].record(stream)
            fq.fq_decode(ctx, nu, codes, rows, out, sp)
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 3:
                enc_ms.append(ev[0].elapsed_time(ev[1]))
                dec_ms.append(ev[1].elapsed_time(ev[2]))
        err = ((out.double() - x64) ** 2).sum(dim=1)
        mse = float((err / xx).mean())
        flags = fq.fq_status(ctx, sp)
        R = fq.fq_record_bits(ctx)
        points.append({"codec": codec, "k": k, "N": N, "bits_per_coordinate": round(np.log2(N) / k, 4),
                       "record_bits": R, "relative_mse": mse,
                       "encode_vectors_per_s": rows / (statistics.median(enc_ms) / 1e3),
                       "decode_vectors_per_s": rows / (statistics.median(dec_ms) / 1e3),
                       "codebook_build_s": round(build_s, 2), "device_flags": flags})
        ctx.close()
        del nu, codes, out
    line = {"metric": "relative MSE E|x - x_hat|^2 / |x|^2 by bits per coordinate", "unit": "ratio",
            "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{rows} N(0,1) fp16 rows, d = {d}, one shared Haar rotation",
                       "codebooks": "scalar: exact Lloyd-Max on the rotated-coordinate law; fibquant: "
                                    "radial-angular initialisation + 10 Lloyd iterations on "
                                    "max(32768, min(131072, 32 N)) source draws",
                       "timing": "median of steps launches, L2 flushed before each encode"},
            "points": points}
    print(json.dumps(line), flush=True)


def run_lloyd(args) -> None:
    """Codebook building for one workload's (kind, d, k, N) and Lloyd budget: the host builder
    (numpy) against the GPU builder (library encoder + fq_centroid_sums), on the same number of
    block draws and on 16 times as many; each codebook's distortion on held-out rows."""
    import torch
    import random_access_kv_gb300 as fq
    from random_access_kv_gb300 import build as fbuild
    from random_access_kv_gb300 import codebook as pcb

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fbuild.build()
    cfg = args.workload
    w = synth.WORKLOADS[cfg]
    d, k, N = w.d, w.k, w.N
    s = synth.kronecker_offset(cfg)
    restarts = [synth.restart_gaussian(cfg, k, r) for r in range(1, w.lloyd_restarts)]
    nb = d // k
    # held-out rows: every block of a row over its norm is a draw of the block source (identity rotation)
    X_test = torch.from_numpy(synth.source_gaussians(cfg, 65536, d, chunk=9).astype(np.float16)).to(dev)
    eye = np.eye(d, dtype=np.float32)

    def heldout(C):
        ctx = fq.fq_codebook_load(C.astype(np.float32), eye, local)
        T = X_test.shape[0]
        nu, codes = fq.alloc_store(ctx, T, dev)
        fq.fq_encode(ctx, X_test, T, nu, codes)
        out = torch.empty((T, d), dtype=torch.float32, device=dev)
        fq.fq_decode_gather_f32(ctx, nu, codes, T, torch.arange(T, device=dev), T, out)
        x = X_test.double()
        rel = ((out.double() - x) ** 2).sum(dim=1) / (x * x).sum(dim=1)
        ctx.close()
        return float(rel.mean()) / nb

    points = []
    t0 = time.perf_counter()
    C, mse = pcb.build(w.codebook_kind, d, k, N, synth.source_gaussians(cfg, w.lloyd_train, d), w.lloyd_iters,
                       restarts, s)
    points.append({"builder": "host numpy", "block_draws": w.lloyd_train, "seconds": round(time.perf_counter() - t0, 3),
                   "train_mse": mse, "heldout_mse": heldout(C)})
    for mult in (1, 16):
        rows = -(-w.lloyd_train * mult // nb)
        X = synth.source_gaussians(cfg, rows, d, chunk=1).astype(np.float16)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        C, mse = pcb.build_gpu(w.codebook_kind, d, k, N, X, w.lloyd_iters, restarts, s, device=local)
        torch.cuda.synchronize(dev)
        points.append({"builder": "gpu", "block_draws": rows * nb, "seconds": round(time.perf_counter() - t0, 3),
                       "train_mse": mse, "heldout_mse": heldout(C)})
    line = {"metric": "codebook build seconds and per-block distortion, host vs GPU Lloyd", "unit": "s",
            "higher_is_better": False, "n_gpus": 1, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "kind": w.codebook_kind, "d": d, "k": k, "N": N,
                       "lloyd_iters": w.lloyd_iters, "restarts": w.lloyd_restarts,
                       "heldout": "65,536 rows, all d/k blocks each (identity rotation)"},
            "points": points}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--attend", action="store_true", help="time fused decode-into-attention")
    ap.add_argument("--rate-sweep", action="store_true",
                    help="relative MSE and throughput against bits per coordinate (scalar k = 1 vs FibQuant)")
    ap.add_argument("--sweep-d", type=int, choices=[64, 96], default=64,
                    help="with --rate-sweep: the head dimension (96 adds the k = 3 Fibonacci-sphere code)")
    ap.add_argument("--lloyd", action="store_true",
                    help="codebook building: host numpy Lloyd against the GPU Lloyd for --workload")
    ap.add_argument("--q-per-group", type=int, default=1,
                    help="with --attend: queries per cached (layer, head) group (grouped-query attention)")
    ap.add_argument("--groups", type=int, default=0,
                    help="with --attend: the first G (layer, head) groups only (a small case for profiling)")
    ap.add_argument("--archive", action="store_true",
                    help="time the iterated-map archive of symbol streams (encode, decode, random access)")
    ap.add_argument("--archive-workload", choices=sorted(synth.ARCHIVE_WORKLOADS), default="document")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=0,
                    help="rows per tensor (a prefix of the workload; a small case for profiling). "
                         "A multiple of the sequence length for the streaming workload.")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.rate_sweep:
        run_rate_sweep(args)
    elif args.lloyd:
        run_lloyd(args)
    elif args.archive:
        run_archive(args)
    elif args.attend:
        run_attend(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
