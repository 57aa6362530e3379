#!/usr/bin/env python3
"""Benchmark: block-sparse GQA attention forward (schedule + attention + combine).

One step = one pass of the whole forward over one batch of synthetic input: the
reverse index and work list (msa_build_schedule) and the attention with its combine
(msa_sparse_attn_fwd), on the MiniMax M3 shape (N = Lkv = 8192, Hq 64, Hkv 4,
D 128, block 128, topK 16) by default.  Inputs are resident in HBM when the timed
region starts; L2 is flushed (a 256 MiB write, then a 256 MiB read that leaves it holding
clean lines) before every timed step, outside the step's events.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the oracle (plain fp64 C on the host cores) on a bounded
sample of the same workload: the pages ship no code, so the oracle is the only
reference implementation there is.  Under torchrun (N > 1) every rank runs its own
independent M3 problem (weak scaling, no collective on the data path); rank 0
prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WINDOW = 2048  # queries per work-list window of the library
METRIC = "sparse-attn fwd useful TFLOP/s and % HBM roofline, M3 shape top16, 1 GB300"
METRIC_BWD = "sparse-attn bwd useful TFLOP/s (dQ, dK, dV; 2.5x the forward's nominal FLOPs), M3 shape top16, 1 GB300"


def kernels_per_step(cfg):
    """Launches of libmsa kernels in one step: schedule (one kernel for tiny inputs: at
    most 1024 list slots, 8192 bitmask words and 8192 segments; else mark, rowscan, one
    fused scan or four scan kernels when there are more than 32768 (window, row)
    segments, scatter + tiles in one launch) + kv_outer + combine + q_outer (the two
    attention kernels not chosen exit at once), plus the E4M3 V widening; where the sizes
    alone fix AUTO's choice (N * Hkv * topK * (10 N - 13) <= 35000 N) only q_outer."""
    rows, words = cfg.Hkv * cfg.nblocks, -(-cfg.N // 32)
    nseg = -(-cfg.N // WINDOW) * rows
    if cfg.N * cfg.Hkv * cfg.topK <= 1024 and rows * words <= 8192 and words <= 64 and nseg <= 8192:
        sched = 1
    else:
        sched = 4 if nseg <= 32768 else 7
    if cfg.N * cfg.Hkv * cfg.topK * (10 * cfg.N - 13) <= 35000 * cfg.N:
        return sched + 1
    return sched + 3 + (1 if cfg.dtype == "e4m3" else 0)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="m3", choices=["tiny", "m3", "long", "lowreuse", "fp8", "decode"])
    ap.add_argument("--lists", default="workload", choices=["workload", "r1", "r4"],
                    help="block lists: the workload's own, or chosen by the R1 / R4 selector (once, before timing)")
    ap.add_argument("--mode", default="general", choices=["general", "tiles", "bwd"],
                    help="general: schedule + attention + combine; tiles: the shared-list forward "
                         "(lists shared by 128 queries for r1, by the workload's query runs otherwise); "
                         "bwd: the backward (dQ, dK, dV) over the forward's schedule, O and LSE")
    ap.add_argument("--partials", default="bf16", choices=["bf16", "fp32"],
                    help="format of the KV-outer partial outputs (the pages' bf16 vs fp32 study)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dispatch-sweep", action="store_true",
                    help="time the step with each path forced over a grid of (dtype, Lkv, N) with uniform "
                         "picks; one JSON line per point (the measurement the AUTO crossover is derived from)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers
def load_peaks(kind="hbm_gbs"):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d[kind]), "measured"
    return (6800.0 if kind == "hbm_gbs" else 1700.0), "fallback"


class L2Flush:
    """Evicts L2 between timed steps: a 256 MiB write, then a 256 MiB read of another buffer.
    The read replaces the written lines, which are dirty and owe a write-back to HBM, with
    clean ones, so that write-back happens here and not inside the next timed step (after a
    write alone, a 327 MB read-only kernel took 68 us instead of 55 us on GB300)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("attn_kv_outer.cu", "ptx.cuh", "msa_internal.h"):
        with open(os.path.join(ROOT, "block_sparse_gqa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """dram read+write bytes per launch of the KV-outer kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"kv_outer_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_hash:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_hash():
        return None
    return int(m.group(1))


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, value, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


# ----------------------------------------------------------------------------- oracle timing
def time_oracle(wl, seconds, seed=0, indices=None):
    """Run the oracle on a seeded query sample sized for ~`seconds` of CPU time.
    Returns (TFLOP/s of useful work, sample description, threads)."""
    import numpy as np
    import oracle
    import workloads
    cfg = wl.cfg
    threads = os.cpu_count() or 1
    Qn, Kn, Vn = wl.np_inputs()
    idx = wl.indices.numpy() if indices is None else indices
    rng = np.random.default_rng(seed)

    def run(nq):
        qids = np.sort(rng.choice(cfg.N, size=nq, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attn_fwd(Qn, Kn, Vn, idx, Lkv=cfg.Lkv, scale=cfg.scale, q_descale=wl.q_descale,
                        k_descale=wl.k_descale, v_descale=wl.v_descale, qids=qids, nthreads=threads)
        return time.perf_counter() - t0

    probe_n = min(16, cfg.N)
    tp = run(probe_n)
    nq = int(min(cfg.N, max(probe_n, probe_n * seconds / max(tp, 1e-6))))
    t = run(nq)
    flops = 4.0 * nq * cfg.Hq * cfg.topK * 128 * cfg.D
    sample = f"{nq} of {cfg.N} queries (seeded uniform sample), all {cfg.Hq} heads, {cfg.name} lists"
    return flops / t / 1e12, sample, threads, t


def time_oracle_bwd(wl, dO_bits, seconds, seed=0):
    """The oracle's backward for the dQ of a seeded query sample sized for ~`seconds`:
    per (query, head) it forms S, dP and dQ over the selected keys, 3 of the 5 products
    of the backward, so the useful FLOPs counted are 6 * nq * Hq * topK * 128 * D."""
    import numpy as np
    import oracle
    cfg = wl.cfg
    threads = os.cpu_count() or 1
    Qn, Kn, Vn = wl.np_inputs()
    idx = wl.indices.numpy()
    rng = np.random.default_rng(seed)

    def run(nq):
        qids = np.sort(rng.choice(cfg.N, size=nq, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attn_bwd(Qn, Kn, Vn, dO_bits, idx, Lkv=cfg.Lkv, scale=cfg.scale, qids=qids, rows=(),
                        nthreads=threads)
        return time.perf_counter() - t0

    probe_n = min(16, cfg.N)
    tp = run(probe_n)
    nq = int(min(cfg.N, max(probe_n, probe_n * seconds / max(tp, 1e-6))))
    t = run(nq)
    flops = 6.0 * nq * cfg.Hq * cfg.topK * 128 * cfg.D
    sample = (f"dQ of {nq} of {cfg.N} queries (seeded uniform sample), all {cfg.Hq} heads, {cfg.name} lists; "
              "S, dP and dQ products counted")
    return flops / t / 1e12, sample, threads, t


# ----------------------------------------------------------------------------- arms
def run_reference(args, world, rank):
    import workloads
    if rank != 0:
        return
    wl = workloads.make_workload(args.workload)
    cfg = wl.cfg
    per_step = max(1.0, min(6.0, 150.0 / max(args.steps + args.warmup, 1)))
    vals, times = [], []
    for k in range(args.warmup + args.steps):
        v, sample, threads, t = time_oracle(wl, per_step, seed=k)
        if k >= args.warmup:
            vals.append(v)
            times.append(t)
    value = statistics.median(vals)
    ms = 1e3 * cfg.nominal_flops() / (value * 1e12)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: N={cfg.N} Lkv={cfg.Lkv} Hq={cfg.Hq} Hkv={cfg.Hkv} D={cfg.D} "
                               f"block=128 topK={cfg.topK}", "reference": "oracle (plain fp64 C, host cores)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample + "; ms_per_step extrapolates the full workload"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_e2e(args, msa, cfg, wl, dev, stream, tiles, lists, tile, descales, flush, pg, world):
    """The step through the public API with host buffers: every step copies its inputs
    (Q, K, V and the block lists) from pinned host memory to the device, runs the
    forward and copies O and LSE back to pinned host memory; all of it is inside the
    timed region.

    Two schedules are timed.  serial: copy in, compute, copy out, one after the other on
    one stream.  pipelined (the reported value): the way a serving loop runs, with two
    device copies of every input and output, the inputs of step k + 1 uploaded on one
    copy stream and the outputs of step k - 1 read back on another while step k
    computes; events order each buffer's reuse.  Per-step inputs (Q alone is 128 MiB at
    the M3 shape) are larger than L2, so the pipelined loop does not flush."""
    import torch

    lists_h = lists.cpu()
    host_in = [t.pin_memory() for t in (wl.Q, wl.K, wl.V, lists_h)]
    o_shape, l_shape = (cfg.N, cfg.Hq, cfg.D), (cfg.N, cfg.Hq)
    host_out = [(torch.empty(o_shape, dtype=torch.bfloat16).pin_memory(),
                 torch.empty(l_shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
    dev_out = [(torch.empty(o_shape, dtype=torch.bfloat16, device=dev),
                torch.empty(l_shape, dtype=torch.float32, device=dev)) for _ in range(2)]
    sched = [None]

    def compute(b):
        dQ, dK, dV, dI = dev_in[b]
        dO, dL = dev_out[b]
        if tiles:
            msa.sparse_attn_fwd_tiles(dQ, dK, dV, dI, tile, scale=cfg.scale, O=dO, LSE=dL)
        else:
            sched[0] = msa.build_schedule(dI, cfg.nblocks, schedule=sched[0])
            msa.sparse_attn_fwd(dQ, dK, dV, sched[0], scale=cfg.scale, O=dO, LSE=dL, descales=descales)

    def upload(b):
        for d, h in zip(dev_in[b], host_in):
            d.copy_(h, non_blocking=True)

    def download(b):
        for h, d in zip(host_out[b], dev_out[b]):
            h.copy_(d, non_blocking=True)

    def serial_step():
        upload(0)
        compute(0)
        download(0)

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def pipelined(nsteps, t0=None, t1=None):
        """Steps 0..nsteps-1 over buffers b = k % 2; t0/t1 bracket the whole run on the
        compute stream (the copy streams start after t0 and the compute stream waits for
        the last read-back before t1)."""
        if t0 is not None:
            t0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for k in range(nsteps):
            b = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(computed[b])  # step k - 2 no longer reads these inputs
                upload(b)
                uploaded[b].record(s_in)
            stream.wait_event(uploaded[b])
            if k >= 2:
                stream.wait_event(downloaded[b])  # step k - 2's outputs have been read back
            compute(b)
            computed[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[b])
                download(b)
                downloaded[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        if t1 is not None:
            t1.record(stream)

    for _ in range(max(3, args.warmup)):
        serial_step()
    pipelined(max(3, args.warmup))
    torch.cuda.synchronize()

    es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(pg)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush()
        es[k].record(stream)
        serial_step()
        ee[k].record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(pg, sum(s.elapsed_time(e) for s, e in zip(es, ee)), dev) / args.steps

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    pipelined(args.steps, t0, t1)
    torch.cuda.synchronize()
    pipe_ms = max_over_ranks(pg, t0.elapsed_time(t1), dev) / args.steps
    if sched[0] is not None:
        st = sched[0].query()
        sched[0].close()
        if st["status"] != 0:
            raise SystemExit(f"device status {st['status']} after the end-to-end steps")

    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    tflops = lambda ms: world * cfg.nominal_flops() / (ms * 1e-3) / 1e12
    return {"value": tflops(pipe_ms), "unit": "TFLOP/s", "ms_per_step": pipe_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "schedule": "pipelined: uploads of step k+1 and read-backs of step k-1 on two copy streams overlap "
                        "step k; double-buffered device inputs and outputs; every step's copies inside one "
                        "timed region",
            "serial": {"value": tflops(serial_ms), "ms_per_step": serial_ms,
                       "schedule": "copy in, compute, copy out on one stream; L2 flushed before each step, "
                                   "outside its events"}}


def run_ours(args, world, rank, local, pg):
    import torch

    import block_sparse_gqa_gb300 as msa
    import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = workloads.CONFIGS[args.workload]
    wl = workloads.make_workload(cfg, seed=cfg.seed + 1000 * rank)
    stream = torch.cuda.current_stream()

    Q, K, V = (t.to(dev) for t in (wl.Q, wl.K, wl.V))
    if args.lists in ("r1", "r4"):
        if cfg.dtype != "bf16":
            raise SystemExit("the selectors take bf16 inputs")
        select = msa.select_blocks_r1 if args.lists == "r1" else msa.select_blocks_r4
        idx_d = select(Q, K, cfg.topK)  # an input of the step, chosen once
        torch.cuda.synchronize()
    else:
        idx_d = wl.indices.to(dev)
    tiles = args.mode == "tiles"
    tstatus = torch.zeros(1, dtype=torch.int32, device=dev)  # device flags of the shared-list kernel
    if tiles:
        tile = 128 if args.lists in ("r1", "r4") else cfg.run
        tile_lists = idx_d[::tile].contiguous()
        if tile % 16 or not torch.equal(torch.repeat_interleave(tile_lists, tile, 0)[:cfg.N], idx_d):
            raise SystemExit(f"workload {cfg.name}: lists are not shared by tiles of a multiple of 16 queries")
    O = torch.empty((cfg.N, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    LSE = torch.empty((cfg.N, cfg.Hq), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    sched = msa.build_schedule(idx_d, cfg.nblocks)
    bwd = args.mode == "bwd"
    if bwd:
        if cfg.dtype != "bf16" or args.lists != "workload":
            raise SystemExit("--mode bwd takes the bf16 workloads with their own lists")
        gen = torch.Generator().manual_seed(cfg.seed + 77 + 1000 * rank)
        dO_h = torch.randn((cfg.N, cfg.Hq, cfg.D), generator=gen).to(torch.bfloat16)
        dO = dO_h.to(dev)
        # the forward whose schedule, O and LSE the backward takes (outside the timed steps)
        msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale, O=O, LSE=LSE)
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # materialise the CUDA event handle
        return evs

    descales = (wl.q_descale, wl.k_descale, wl.v_descale)

    def step(stage):
        if bwd:
            msa.sparse_attn_bwd(Q, K, V, O, dO, LSE, sched, scale=cfg.scale, dQ=dQ, dK=dK, dV=dV,
                                stage_events=[e.cuda_event for e in stage] if stage else None)
            return
        if tiles:
            if stage:
                stage[0].record(stream)
            msa.sparse_attn_fwd_tiles(Q, K, V, tile_lists, tile, scale=cfg.scale, O=O, LSE=LSE, status=tstatus)
            if stage:
                stage[1].record(stream)
                stage[2].record(stream)
            return
        msa.build_schedule(idx_d, cfg.nblocks, schedule=sched)
        msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale, O=O, LSE=LSE, descales=descales,
                            stage_events=[e.cuda_event for e in stage] if stage else None,
                            partials_fp32=args.partials == "fp32")

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    info = sched.query()
    assert info["status"] == 0, info
    kv_path = info["path"] == 1 or tiles or bwd  # else the Q-outer kernel runs (inside the third stage)

    starts, ends = new_events(args.steps), new_events(args.steps)
    stages = [new_events(3) for _ in range(args.steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(pg)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    for k in range(args.steps):
        flush()
        starts[k].record(stream)
        step(None)
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    clock_info = clocks.stop()
    # stage times come from a second pass of the same steps with events between the stages:
    # an event recorded between two kernels ends their programmatic launch overlap, so the
    # timed pass above records none
    sstarts = new_events(args.steps)
    for k in range(args.steps):
        flush()
        sstarts[k].record(stream)
        step(stages[k])
    torch.cuda.synchronize()
    after = sched.query()  # the device's sticky flags after the timed steps
    if tiles:
        after = {"status": int(tstatus.item())}
    if after["status"] != 0:
        raise SystemExit(f"device status {after['status']} after the timed steps (1 bad index, 2 wait timed out)")

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    attn_ms = [st[0].elapsed_time(st[1]) for st in stages]
    comb_ms = [st[1].elapsed_time(st[2]) for st in stages]
    sched_ms = [s.elapsed_time(st[0]) for s, st in zip(sstarts, stages)]
    total_ms = max_over_ranks(pg, sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    nominal = cfg.nominal_flops() * (2.5 if bwd else 1.0)  # the backward runs 5 products to the forward's 2
    value = world * nominal / (ms_per_step * 1e-3) / 1e12

    # algorithmic bytes: the KV-outer kernel reads Q once, each selected K/V block once, the
    # lists and tiles, and writes every partial row and its (m, l) once; the whole step adds
    # the combine (partials read, O and LSE written) and the schedule's list reads
    E, nsb, T = info["entries"], info["nsb"], info["ntiles"]
    G, D = cfg.G, cfg.D
    es = 1 if cfg.dtype == "e4m3" else 2  # bytes per input element
    q_bytes = cfg.N * cfg.Hq * D * es
    kv_bytes = nsb * 2 * 128 * D * es
    part_bytes = E * G * ((4 if args.partials == "fp32" else 2) * D + 8)  # partial row + float2 (m, l)
    meta_attn = E * 4 + T * 16
    attn_bytes = q_bytes + kv_bytes + part_bytes + meta_attn
    comb_bytes = part_bytes + cfg.N * cfg.Hkv * cfg.topK * 4 + cfg.N * cfg.Hq * (2 * D + 4)
    step_bytes = attn_bytes + comb_bytes + cfg.N * cfg.Hkv * cfg.topK * 4 * 3
    peak, peak_kind = load_peaks()
    attn_mean = statistics.mean(attn_ms)
    achieved = attn_bytes / (attn_mean * 1e-3) / 1e9
    traffic = recorded_traffic(cfg.name) if args.partials == "bf16" else None  # profiled with bf16 partials
    if not kv_path:
        # Q-outer: Q once, each distinct selected K/V block once (the pages' deduplicated
        # bytes), the block lists, O and LSE written; timed in the combine stage, where the
        # Q-outer kernel runs (the combine launch exits at once)
        attn_bytes = q_bytes + kv_bytes + cfg.N * cfg.Hkv * cfg.topK * 4 + cfg.N * cfg.Hq * (2 * D + 4)
        attn_mean = statistics.mean(comb_ms)
        achieved = attn_bytes / (attn_mean * 1e-3) / 1e9
        traffic = None
        step_bytes = attn_bytes + cfg.N * cfg.Hkv * cfg.topK * 4 * 3
    roof = {"kernel": "kv_outer_kernel" if kv_path else "q_outer_kernel", "bound": "hbm", "achieved": achieved,
            "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": traffic, "algorithmic_bytes": attn_bytes,
            "peak_source": f"{peak_kind} MEASURED_PEAKS.json hbm_gbs" if peak_kind == "measured"
            else "fallback 6.8 TB/s", "launch_ms": attn_mean}
    if tiles:
        # the shared-list kernel moves Q, the distinct K/V blocks (re-read from L2 per
        # 16-query pair) and O: it is bound by the tensor pipe and the softmax, not HBM
        flops = 4.0 * 128 * D * G * E
        tpeak, tkind = load_peaks("bf16_tflops_sustained")
        achieved_t = flops / (attn_mean * 1e-3) / 1e12
        roof = {"kernel": "tiles_kernel", "bound": "tensor", "achieved": achieved_t, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved_t / tpeak, "traffic": None, "algorithmic_flops": flops,
                "peak_source": f"{tkind} MEASURED_PEAKS.json bf16_tflops_sustained", "launch_ms": attn_mean}
        step_bytes = q_bytes + kv_bytes + cfg.N * cfg.Hq * (2 * D + 4) + tile_lists.numel() * 4
    if bwd:
        # the KV-stationary backward kernel: five 128 x 128 x 128 products per tile (S, dP,
        # dV, dK, dQ) over the selected pairs; bound by the tensor pipe and the chain
        # between them.  Step bytes: Q, dO and O read once, LSE and D, the selected K/V
        # blocks, the dQ contributions written and re-read, the units' fp32 dK/dV written
        # and re-read, dQ, dK, dV written, the lists.
        flops = 10.0 * 128 * D * G * E
        tpeak, tkind = load_peaks("bf16_tflops_sustained")
        achieved_t = flops / (attn_mean * 1e-3) / 1e12
        roof = {"kernel": "bwd_kv_kernel", "bound": "tensor", "achieved": achieved_t, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved_t / tpeak, "traffic": None, "algorithmic_flops": flops,
                "peak_source": f"{tkind} MEASURED_PEAKS.json bf16_tflops_sustained", "launch_ms": attn_mean}
        counts = sched.export()["counts"]
        units = int(((counts + 255) // 256).sum())
        step_bytes = (3 * q_bytes + cfg.N * cfg.Hq * 12 + kv_bytes + 2 * E * G * D * 2 + 2 * units * 2 * 128 * D * 4
                      + q_bytes + 2 * cfg.Lkv * cfg.Hkv * D * 2 + E * 4 + cfg.N * cfg.Hkv * cfg.topK * 4)

    e2e = None
    if not args.no_e2e and not bwd:
        e2e = time_e2e(args, msa, cfg, wl, dev, stream, tiles, tile_lists if tiles else idx_d,
                       tile if tiles else None, descales, flush, pg, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and bwd:
        v, sample, threads, _ = time_oracle_bwd(wl, dO_h.view(torch.int16).numpy().view("uint16"), args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample, threads, _ = time_oracle(wl, args.cpu_seconds, indices=idx_d.cpu().numpy())
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample}

    sched.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)" if es == 1 else "bf16",
        "data": f"synthetic (seeded N(0,1) Q/K/V{', per-tensor E4M3' if es == 1 else ''}, {cfg.picks} block picks)",
        "config": {"workload": f"{cfg.name}: N={cfg.N} Lkv={cfg.Lkv} Hq={cfg.Hq} Hkv={cfg.Hkv} D={cfg.D} block=128 "
                               f"topK={cfg.topK}, causal, own block + up to {cfg.topK - 1} {cfg.picks} earlier blocks",
                   "l2": "flushed before every timed step, outside the step events: a 256 MiB write, then a 256 MiB read that replaces the written (dirty) lines with clean ones, so their write-back to HBM is not inside the step",
                   "stage_timing": "stage_ms and roofline.launch_ms from a second pass of the same steps with "
                                   "events between the stages (the timed pass records none: an event between two "
                                   "kernels ends their programmatic launch overlap)",
                   "parallelism": f"independent problem per GPU x{world}",
                   "path": "bwd" if bwd else "tiles" if tiles else ("kv_outer" if kv_path else "q_outer"),
                   "lists": (f"{args.lists.upper()} selector (chosen once, before timing)" if args.lists != "workload"
                             else "workload"),
                   "partials": args.partials,
                   "entries": E, "nsb": nsb, "tiles": T},
        "roofline": roof,
        "path_roofline": {"bytes_per_step": step_bytes, "achieved_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
                          "frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak},
        "stage_ms": ({"prep+units": statistics.mean(sched_ms), "bwd_kv": statistics.mean(attn_ms),
                      "reduce+dq": statistics.mean(comb_ms)} if bwd else
                     {"schedule": statistics.mean(sched_ms), "attention": statistics.mean(attn_ms),
                      "combine": statistics.mean(comb_ms)} if kv_path or tiles else
                     {"schedule": statistics.mean(sched_ms), "kv_outer_exit": statistics.mean(attn_ms),
                      "combine_exit+q_outer": statistics.mean(comb_ms)}),
        "selected_pair_tflops": world * (10.0 if bwd else 4.0) * 128 * D * G * E / (ms_per_step * 1e-3) / 1e12,
        "gpu_launches": (5 if bwd else 1 if tiles else kernels_per_step(cfg)) * args.steps,
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# (dtype, Lkv, Hkv, topK, query counts)
SWEEP_GRID = [("bf16", 16384, 4, 16, (1, 16, 64, 128, 256, 512, 1024, 2048, 4096)),
              ("bf16", 131072, 4, 16, (1, 16, 64, 128, 256, 512, 1024, 2048, 4096)),
              ("bf16", 524288, 4, 16, (1, 16, 64, 128, 256, 512, 1024, 2048)),
              ("e4m3", 131072, 4, 16, (1, 16, 64, 128, 256, 512, 1024, 2048, 4096)),
              ("bf16", 131072, 2, 8, (16, 64, 128, 256, 512, 1024)),
              ("bf16", 131072, 8, 32, (4, 16, 32, 64, 128, 256)),
              ("bf16", 32768, 1, 4, (64, 256, 512, 1024, 2048))]


def run_dispatch_sweep(args):
    """Step time (schedule + forward, L2 flushed before each step) with the path forced to
    KV-outer and to Q-outer, over queries at the tail of contexts of several lengths
    (Hq = 16 Hkv, D 128, own block + topK - 1 uniform earlier blocks).  Q / K / V are
    drawn on the device (seeded): only the timing is used, and the lists are the seeded
    uniform ones of the workloads module.  One JSON line per (dtype, Lkv, N)."""
    import torch

    import block_sparse_gqa_gb300 as msa
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    gen = torch.Generator(device=dev)
    for dtype, Lkv, Hkv, topK, Ns in SWEEP_GRID:
        gen.manual_seed(Lkv)
        K = torch.randn((Lkv, Hkv, 128), generator=gen, device=dev)
        V = torch.randn((Lkv, Hkv, 128), generator=gen, device=dev)
        if dtype == "e4m3":
            K, V = (x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8) for x in (K, V))
        else:
            K, V = K.to(torch.bfloat16), V.to(torch.bfloat16)
        for N in Ns:
            cfg = workloads.Config("sweep", N, Lkv, 16 * Hkv, Hkv, 128, topK, "uniform", 2000 + N, dtype=dtype)
            idx = torch.from_numpy(workloads.make_indices(cfg)).to(dev)
            Q = torch.randn((N, 16 * Hkv, 128), generator=gen, device=dev)
            Q = Q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8) if dtype == "e4m3" else Q.to(torch.bfloat16)
            O = torch.empty((N, 16 * Hkv, 128), dtype=torch.bfloat16, device=dev)
            LSE = torch.empty((N, 16 * Hkv), dtype=torch.float32, device=dev)
            sched = msa.build_schedule(idx, cfg.nblocks)
            desc = (1.0, 1.0, 1.0)
            row = {"dtype": dtype, "Lkv": Lkv, "Hkv": Hkv, "topK": topK, "N": N}
            for path in ("kv_outer", "q_outer"):
                def step():
                    msa.build_schedule(idx, cfg.nblocks, schedule=sched)
                    msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale, O=O, LSE=LSE, path=path, descales=desc)
                for _ in range(args.warmup):
                    step()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.steps)]
                torch.cuda.synchronize()
                for a, b in evs:
                    flush()
                    a.record(stream)
                    step()
                    b.record(stream)
                torch.cuda.synchronize()
                row[path + "_us"] = 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)
            info = sched.query()
            assert info["status"] == 0, info
            sched.close()
            row.update(nsb=info["nsb"], entries=info["entries"], nsb_per_N=info["nsb"] / N,
                       auto=("kv_outer" if info["path"] == 1 else "q_outer"),
                       faster=("kv_outer" if row["kv_outer_us"] <= row["q_outer_us"] else "q_outer"))
            print(json.dumps(row), flush=True)


def main():
    args = parse_args()
    if args.dispatch_sweep:
        run_dispatch_sweep(args)
        return
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work or collectives
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local, pg = dist_setup(args)
    run_ours(args, world, rank, local, pg)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
