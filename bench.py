#!/usr/bin/env python3
"""Benchmark of the SparseLoCo pseudo-gradient codec on GB300.

One step is one round of the codec's hot path on one GPU:
  1. spl_ef_compress on 2^30 fp32 pseudo-gradient values (Laplace(0, 1e-4), beta 0.95,
     fp32 error buffer carried over the rounds; a fresh pseudo-gradient each round, cycling
     through ten held in HBM): 262,144 chunks -> 262,144 records of 112 B + 262,144 scales;
  2. spl_decode_aggregate of 24 peers' records of a 2^30-value tensor into the fp32 mean,
     fused with the outer step theta <- theta - 0.7 * mean.
The metric is algorithmic HBM bytes of the step per second (GB/s): compress moves
12 n + 116 C bytes (read delta and e, write e, records and scales), decode moves
24 x 116 C + 12 n bytes (read records and scales, write the mean, read and write theta).

Arms:
  default            the CUDA library; prints one JSON line (rank 0).
  --impl reference   the CPU oracle timed on the host cores on a bounded sample of the same
                     workload (the only other place this script runs the oracle).

Multi-GPU (python -m torch.distributed.run ... bench.py --gpus N): every rank runs the whole
step on its own peer's data (independent problems, no collective on the data path); the
time is the max over ranks and the value is the sum of all ranks' bytes over that time.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "EF-compress and decode-aggregate GB/s on 1 GB300; % of HBM roofline; vs CPU oracle"
N_ELEMS = 1 << 30
CHUNK = 4096
RECORD = 112
PEERS = 24
ROUNDS = 10          # distinct pseudo-gradients, one per round, cycled over the steps
BETA = 0.95
LR = 0.7
N_CHUNKS = (N_ELEMS + CHUNK - 1) // CHUNK
WORKLOAD = ("EF-compress of 2^30 fp32 Laplace(0,1e-4) values (beta 0.95, fp32 error buffer "
            "carried over the rounds, a fresh delta each round from 10 held in HBM) + "
            "decode-aggregate of 24 peers' records into a 2^30 fp32 mean fused with outer "
            "SGD (lr 0.7) on fp32 theta ~ N(0,0.02)")
FALLBACK_HBM_GBS = 6800.0


def compress_bytes(n: int, C: int, record: int = RECORD) -> int:
    return 12 * n + (record + 4) * C


def decode_bytes(n: int, C: int, P: int, theta: bool = True, record: int = RECORD) -> int:
    return P * (record + 4) * C + 4 * n + (8 * n if theta else 0)


# The codec variants timed by --workload codecs: (chunk length, k, scale rule), the default
# codec first.
CODECS = [(4096, 64, 0), (4096, 64, 1), (4096, 32, 0), (4096, 32, 1), (4096, 128, 0),
          (4096, 128, 1), (2048, 32, 0), (2048, 32, 1), (8192, 128, 0), (8192, 128, 1)]



# ---------------------------------------------------------------------------------------------
# Distributed helpers (one process per GPU; NCCL on GPUs, gloo on CPU)
# ---------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed_base(rank: int) -> int:
    """Seed block of a rank's peer: the rounds' deltas at base + 10000 r (r < 10), its 24
    peers' deltas at base + 1..24, theta at base + 5000; blocks of different ranks never
    overlap."""
    return 1 + 100000 * rank


def round_seeds(base: int) -> list[int]:
    return [base + 10000 * r for r in range(ROUNDS)]


def aggregate_value(bytes_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: all ranks' bytes over the slowest rank's time."""
    return bytes_per_rank * world / max_seconds / 1e9


# ---------------------------------------------------------------------------------------------
# Peaks, clocks and the committed DRAM-traffic figure
# ---------------------------------------------------------------------------------------------
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name: str) -> str:
    """Hash of a kernel's code: its launch unit, its template header, the device helpers and
    the launch constants, with // comments and blank lines left out (a comment edit does not
    change the kernel)."""
    src = os.path.join(ROOT, "compressed_pseudo_gradient_gb300", "csrc")
    h = hashlib.sha256()
    for f in (f"{name}.cu", f"{name}.cuh", "spl_device.cuh", "spl_kernels.h"):
        with open(os.path.join(src, f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def smi_id(dev) -> str:
    """nvidia-smi -i identifier of a torch device (its UUID, else its ordinal)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index)


class ClockSampler:
    """nvidia-smi clock/throttle samples every `interval_ms` while the timed region runs.

    Entering starts nvidia-smi and waits (up to 5 s) for its first sample, so that the timed
    region that follows is covered from its start.  Only samples whose own timestamp lies
    between entering and leaving count (nvidia-smi's output reaches the pipe in bursts, so
    arrival times say little)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 10):
        self.gpu = gpu_id
        self.interval = interval_ms
        self.proc = None
        self.lines = []          # (arrival time, line)
        self.t_in = self.t_out = None
        self._first = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            self._first.wait(timeout=5.0)
        except OSError:
            self.proc = None
        self.t_in = datetime.datetime.now()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self._first.set()

    def __exit__(self, *exc):
        self.t_out = datetime.datetime.now()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t_in is None or t < self.t_in or (self.t_out is not None and t > self.t_out):
                    continue
                sm.append(float(parts[2]))
                mx = float(parts[3])
            except ValueError:
                continue
            for name, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "interval_ms": self.interval}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "interval_ms": self.interval}


# ---------------------------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------------------------
def setup_workload(dev, seed_base: int, n: int):
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    from compressed_pseudo_gradient_gb300 import synth

    C = (n + CHUNK - 1) // CHUNK
    buf = {"n": n}
    buf["deltas"] = [synth.laplace(n, 1e-4, synth.generator(sd, dev), dev)
                     for sd in round_seeds(seed_base)]
    buf["delta"] = buf["deltas"][0]
    buf["round"] = 0
    buf["ef"] = torch.zeros(n, dtype=torch.float32, device=dev)
    buf["payload"] = torch.empty((C, RECORD), dtype=torch.uint8, device=dev)
    buf["scales"] = torch.empty(C, dtype=torch.float32, device=dev)
    peers_pl, peers_sc = [], []
    tmp_e = torch.empty(n, dtype=torch.float32, device=dev)
    for p in range(PEERS):
        d = synth.laplace(n, 1e-4, synth.generator(seed_base + 1 + p, dev), dev)
        tmp_e.zero_()
        pl, sc = spl.ef_compress(d, tmp_e, BETA)
        peers_pl.append(pl)
        peers_sc.append(sc)
        del d
    del tmp_e
    buf["peers_pl"], buf["peers_sc"] = peers_pl, peers_sc
    buf["theta"] = synth.theta(n, synth.generator(seed_base + 5000, dev), dev)
    buf["mean"] = torch.empty(n, dtype=torch.float32, device=dev)
    buf["flags"] = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return buf


def gpu_step(buf, ev=None):
    """One round: compress, then decode-aggregate with the fused outer step.  With `ev`
    (four events), records compress start/end and decode start/end on the current stream."""
    import compressed_pseudo_gradient_gb300 as spl
    if ev:
        ev[0].record()
    delta = buf["deltas"][buf["round"] % ROUNDS]   # this round's pseudo-gradient
    buf["round"] += 1
    spl.ef_compress(delta, buf["ef"], BETA, payload=buf["payload"], scales=buf["scales"],
                    flags=buf["flags"])
    if ev:
        ev[1].record()
        ev[2].record()
    spl.decode_aggregate(buf["peers_pl"], buf["peers_sc"], buf["n"], mean=buf["mean"],
                         theta=buf["theta"], lr=LR, flags=buf["flags"], stats=buf.get("stats"))
    if ev:
        ev[3].record()
    return 2   # kernels launched


def host_link_gbs(dev, nbytes: int = 1 << 30) -> float:
    """Measured host-link bandwidth with both directions busy: a pinned H2D and a D2H copy of
    nbytes each on two streams at once; (2 nbytes) / time of the slower, best of 3."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = 0.0
    for _ in range(3):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)
        torch.cuda.synchronize(dev)
        best = max(best, 2 * nbytes / (time.perf_counter() - t0) / 1e9)
    return best


def run_offload(args, dev):
    """Compress of the 2^30-value Laplace workload with the error buffer in pinned host
    memory: the buffer's 8 bytes per value cross the host link, delta stays in HBM."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    from compressed_pseudo_gradient_gb300 import synth

    n = args.elements
    C = (n + CHUNK - 1) // CHUNK
    delta = synth.laplace(n, 1e-4, synth.generator(1, dev), dev)
    ef = torch.zeros(n, dtype=torch.float32).pin_memory()
    payload = torch.empty((C, RECORD), dtype=torch.uint8, device=dev)
    scales = torch.empty(C, dtype=torch.float32, device=dev)
    link = host_link_gbs(dev)
    for _ in range(args.warmup):
        spl.ef_compress(delta, ef, BETA, payload=payload, scales=scales)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        spl.ef_compress(delta, ef, BETA, payload=payload, scales=scales)
    end.record()
    torch.cuda.synchronize(dev)
    secs = start.elapsed_time(end) / 1e3 / args.steps
    link_bytes = 8 * n
    line = {"metric": METRIC, "value": round(compress_bytes(n, C) / secs / 1e9, 2),
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "offload: compress 2^30 fp32 with the error buffer in pinned "
                                   "host memory", "n": n,
                       "host_link": {"bytes_per_step": link_bytes,
                                     "achieved_gbs": round(link_bytes / secs / 1e9, 1),
                                     "measured_peak_gbs": round(link, 1),
                                     "frac": round(link_bytes / secs / 1e9 / link, 4)}},
            "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)
    return 0


def setup_other_workload(name: str, dev, layer_scale: int = 1):
    """Buffers and one-round step of another workload, a fresh pseudo-gradient each round (the
    workload's round count of them, cycled).  heavy_tail_bf16: 2^27 bf16 compress + 8-peer mean;
    decoder_layer: the 72B-class layer's nine tensors compressed in one multi-tensor call;
    tiny: 2^20 compress + 4-peer mean.  Returns (step, info): step(r, ev=None) runs round r and,
    given three events, records them before the compress, between the kernels and after the
    decode; info holds the sizes and the algorithmic bytes of each kernel."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    from compressed_pseudo_gradient_gb300 import synth

    wl = synth.WORKLOADS[name]
    R = wl.rounds
    if wl.name == "decoder_layer":
        shapes = tuple((nm, (max(1, sh[0] // layer_scale),) + tuple(sh[1:]))
                       for nm, sh in synth.DECODER_LAYER_SHAPES)
        rounds = [synth.decoder_layer_round(synth.generator(1 + 1000 * r, dev), dev, shapes)
                  for r in range(R)]
        efs = [torch.zeros_like(d) for d in rounds[0]]
        sizes = [d.numel() for d in rounds[0]]
        C = sum((k + CHUNK - 1) // CHUNK for k in sizes)
        payload = torch.empty((C, RECORD), dtype=torch.uint8, device=dev)
        scales = torch.empty(C, dtype=torch.float32, device=dev)
        comp_bytes = sum(compress_bytes(k, (k + CHUNK - 1) // CHUNK) for k in sizes)

        def step(r, ev=None):
            if ev:
                ev[0].record()
            spl.ef_compress_multi(rounds[r % R], efs, wl.beta, payload=payload, scales=scales)
            if ev:
                ev[1].record()
                ev[2].record()
            return 1
        name = wl.name if layer_scale == 1 else f"{wl.name} (rows / {layer_scale})"
        return step, {"name": name, "n": sum(sizes), "chunks": C, "rounds": R, "peers": 0,
                      "dtype": "f32", "comp_bytes": comp_bytes, "dec_bytes": 0,
                      "tensors": len(sizes)}
    n = wl.n
    C = (n + CHUNK - 1) // CHUNK
    rounds = [synth.delta_round(wl, synth.generator(1 + 1000 * r, dev), dev) for r in range(R)]
    ef = torch.zeros(n, dtype=torch.float32, device=dev)
    payload = torch.empty((C, RECORD), dtype=torch.uint8, device=dev)
    scales = torch.empty(C, dtype=torch.float32, device=dev)
    pls, scs = [], []
    tmp = torch.empty(n, dtype=torch.float32, device=dev)
    for p in range(wl.peers):
        d = synth.delta_round(wl, synth.generator(2 + p, dev), dev)
        tmp.zero_()
        pl, sc = spl.ef_compress(d, tmp, wl.beta)
        pls.append(pl)
        scs.append(sc)
    del tmp
    mean = torch.empty(n, dtype=torch.float32, device=dev)
    esz = 2 if rounds[0].dtype == torch.bfloat16 else 4
    comp_bytes = (esz + 8) * n + (RECORD + 4) * C

    def step(r, ev=None):
        if ev:
            ev[0].record()
        spl.ef_compress(rounds[r % R], ef, wl.beta, payload=payload, scales=scales)
        if ev:
            ev[1].record()
        spl.decode_aggregate(pls, scs, n, mean=mean)
        if ev:
            ev[2].record()
        return 2
    return step, {"name": wl.name, "n": n, "chunks": C, "rounds": R, "peers": wl.peers,
                  "dtype": "bf16" if esz == 2 else "f32", "comp_bytes": comp_bytes,
                  "dec_bytes": decode_bytes(n, C, wl.peers, theta=False)}


def time_steps(dev, run_round, steps: int, ev_count: int = 0):
    """Seconds for `steps` calls of run_round(k[, events]) between two CUDA events on the
    current stream, with per-step events when ev_count > 0 (returned as lists)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ev_count)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record()
    for k in range(steps):
        if ev_count:
            run_round(k, evs[k])
        else:
            run_round(k)
    end.record()
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end) / 1e3, evs


def kernel_split(info, evs, peak):
    """Per-kernel averages from three events per step: compress, then decode."""
    out = {}
    c_s = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    gbs = info["comp_bytes"] / c_s / 1e9
    out["ef_compress"] = {"ms": round(1e3 * c_s, 4), "GB/s": round(gbs, 1),
                          "frac_of_hbm": round(gbs / peak, 4),
                          "Gelem/s": round(info["n"] / c_s / 1e9, 2)}
    if info["dec_bytes"]:
        d_s = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / 1e3
        gbs = info["dec_bytes"] / d_s / 1e9
        out["decode_aggregate"] = {"ms": round(1e3 * d_s, 4), "GB/s": round(gbs, 1),
                                   "frac_of_hbm": round(gbs / peak, 4),
                                   "Gelem/s": round(info["n"] / d_s / 1e9, 2)}
    return out


def movement_record(dev, n: int, C: int, steps: int, warmup: int, comp_ms: float,
                    dec_ms: float):
    """Each kernel against its own data movement: the library's reference kernels
    (spl_calib_moves) move the sender's and the receiver's dense bytes (12 B per value) the
    way the kernels do, in their order of chunks, with none of the codec's arithmetic; scaled
    to each kernel's algorithmic bytes (records and scales included) at the same rate, that
    time is the floor the kernel's own access pattern sets.  Mean of `steps` after `warmup`."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    a = torch.rand(n, device=dev)
    b = torch.rand(n, device=dev)
    c = torch.empty(n, device=dev)
    d = torch.empty(n, device=dev)
    runs = {"sender": lambda: spl.calib_moves(spl.CALIB_SENDER_MOVES, a, b, out0=c),
            "receiver": lambda: spl.calib_moves(spl.CALIB_RECEIVER_MOVES, a, out0=c, out1=d)}
    out = {}
    for name, fn in runs.items():
        for _ in range(warmup):
            fn()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s0.record()
        for _ in range(steps):
            fn()
        s1.record()
        torch.cuda.synchronize(dev)
        out[name] = s0.elapsed_time(s1) / steps
    del a, b, c, d
    torch.cuda.empty_cache()
    comp_floor = out["sender"] * compress_bytes(n, C) / (12 * n)
    dec_floor = out["receiver"] * decode_bytes(n, C, PEERS) / (12 * n)
    return {"sender_moves_ms": round(out["sender"], 4),
            "receiver_moves_ms": round(out["receiver"], 4),
            "ef_compress": {"floor_ms": round(comp_floor, 4),
                            "frac_of_own_movement": round(comp_floor / comp_ms, 4)},
            "decode_aggregate": {"floor_ms": round(dec_floor, 4),
                                 "frac_of_own_movement": round(dec_floor / dec_ms, 4)},
            "note": "spl_calib_moves in the kernels' order of chunks; floor = its time scaled "
                    "to the kernel's algorithmic bytes"}


def other_workload_record(name: str, dev, steps: int, warmup: int):
    """A sub-record of the default line: `steps` rounds of another workload as plain calls,
    timed as a whole and per kernel, with the clocks sampled meanwhile."""
    import torch
    step, info = setup_other_workload(name, dev)
    warm_secs, _ = time_steps(dev, step, warmup)
    # at least 0.25 s of timed steps, so the clock samples cover the region several times
    steps = int(min(2000, max(steps, math.ceil(0.25 / (warm_secs / warmup)))))
    with ClockSampler(smi_id(dev)) as clk:
        secs, evs = time_steps(dev, step, steps, ev_count=3)
    peak, _ = read_peaks()
    step_bytes = info["comp_bytes"] + info["dec_bytes"]
    value = step_bytes * steps / secs / 1e9
    rec = {"workload": info["name"], "n": info["n"], "chunks": info["chunks"],
           "dtype": info["dtype"], "rounds": info["rounds"], "peers": info["peers"],
           "steps": steps, "ms_per_step": round(1e3 * secs / steps, 4),
           "step_bytes": step_bytes, "GB/s": round(value, 1),
           "frac_of_hbm": round(value / peak, 4)}
    rec.update(kernel_split(info, evs, peak))
    rec["clocks"] = clk.summary()
    del step
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return rec


def run_other_workload(args, dev):
    """Times one round of another workload (same metric: algorithmic bytes per second), as
    plain calls and as CUDA graphs of each round replayed in turn; reports the faster."""
    import torch

    step, info = setup_other_workload(args.workload, dev, args.layer_scale)
    R = info["rounds"]
    step_bytes = info["comp_bytes"] + info["dec_bytes"]
    for k in range(args.warmup):
        step(k)
    peak, kind = read_peaks()
    with ClockSampler(smi_id(dev)) as clk:
        eager_secs, evs = time_steps(dev, step, args.steps, ev_count=3)
    split = kernel_split(info, evs, peak)
    launches = step(0) * args.steps
    # each round's step captured once into a CUDA graph and replayed in turn: the calls are
    # stream-ordered and never allocate or synchronise, so a launch-bound step sheds its
    # per-call host cost
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step(0)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(r)
        graphs.append(g)
    for k in range(args.warmup):
        graphs[k % R].replay()
    graph_secs, _ = time_steps(dev, lambda k: graphs[k % R].replay(), args.steps)
    # the faster launch mode is the one a user would take: graphs pay off where launches bound
    # the step (tiny), plain calls where the kernels do
    use_graph = graph_secs < eager_secs
    secs = graph_secs if use_graph else eager_secs
    other = eager_secs if use_graph else graph_secs
    value = step_bytes * args.steps / secs / 1e9
    cfg = {"workload": info["name"], "n": info["n"], "rounds": R, "step_bytes": step_bytes,
           "frac_of_hbm": round(value / peak, 4), "peak_kind": kind,
           "launch": "CUDA graph of the step, replayed" if use_graph else "plain calls",
           "other_launch_ms_per_step": round(1e3 * other / args.steps, 4)}
    cfg.update(split)
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": info["dtype"], "data": "synthetic",
            "config": cfg, "clocks": clk.summary(), "gpu_launches": launches}
    print(json.dumps(line), flush=True)
    return 0


def run_codecs(args, dev):
    """Times the receive step (compress of n fp32 Laplace(0,1e-4) values with beta 0.95, then
    the 24-peer decode fused with the outer step) for the default codec and each variant;
    one JSON line with a per-codec breakdown.  The value is all codecs' bytes over their
    total time."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    from compressed_pseudo_gradient_gb300 import synth

    n = args.elements
    delta = synth.laplace(n, 1e-4, synth.generator(1, dev), dev)
    ef = torch.zeros(n, dtype=torch.float32, device=dev)
    theta = synth.theta(n, synth.generator(5000, dev), dev)
    mean = torch.empty(n, dtype=torch.float32, device=dev)
    tmp = torch.empty(n, dtype=torch.float32, device=dev)
    peak, kind = read_peaks()
    rows, total_bytes, total_s, launches = [], 0, 0.0, 0
    for codec in CODECS:
        L = codec[0]
        C = (n + L - 1) // L
        rb = spl.record_bytes(codec)
        payload = torch.empty((C, rb), dtype=torch.uint8, device=dev)
        scales = torch.empty(C, dtype=torch.float32, device=dev)
        pls, scs = [], []
        for p in range(PEERS):
            d = synth.laplace(n, 1e-4, synth.generator(2 + p, dev), dev)
            tmp.zero_()
            pl, sc = spl.ef_compress(d, tmp, BETA, codec=codec)
            pls.append(pl)
            scs.append(sc)
            del d
        ef.zero_()

        def step(ev=None):
            if ev:
                ev[0].record()
            spl.ef_compress(delta, ef, BETA, payload=payload, scales=scales, codec=codec)
            if ev:
                ev[1].record()
            spl.decode_aggregate(pls, scs, n, mean=mean, theta=theta, lr=LR, codec=codec)
            if ev:
                ev[2].record()
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for k in range(args.steps):
            step(evs[k])
            launches += 2
        torch.cuda.synchronize(dev)
        c_s = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) / 1e3
        d_s = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / 1e3
        cb, db = compress_bytes(n, C, rb), decode_bytes(n, C, PEERS, record=rb)
        total_bytes += (cb + db) * args.steps
        total_s += (c_s + d_s) * args.steps
        rows.append({"codec": {"chunk": codec[0], "topk": codec[1],
                               "scale": "mean_abs" if codec[2] else "max_abs"},
                     "record_bytes": rb,
                     "ef_compress": {"ms": round(1e3 * c_s, 4), "GB/s": round(cb / c_s / 1e9, 1),
                                     "frac_of_hbm": round(cb / c_s / 1e9 / peak, 4)},
                     "decode_aggregate": {"ms": round(1e3 * d_s, 4),
                                          "GB/s": round(db / d_s / 1e9, 1),
                                          "frac_of_hbm": round(db / d_s / 1e9 / peak, 4)}})
        del pls, scs, payload, scales
        torch.cuda.empty_cache()
    value = total_bytes / total_s / 1e9
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total_s / args.steps / len(CODECS), 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"codec variants: receive step at {n} values, 24 peers",
                       "n": n, "peak_gbs": peak, "peak_kind": kind, "codecs": rows},
            "gpu_launches": launches}
    print(json.dumps(line), flush=True)
    return 0


def run_hbm_mix(args, dev):
    """Context for the roofline: what plain streaming torch kernels reach on this GPU for the
    two kernels' read/write mixes, on 2^30 fp32 values each, best of `steps` (CUDA events):
    a copy (4 B read + 4 B written per value, the measured peak's own kernel), an add (8 + 4,
    the compress's mix: delta and the error buffer in, the error buffer out), frexp (4 + 8,
    the decode's mix: theta in, the mean and theta out) and a fill (0 + 4, the mix of a
    mean-only decode, whose few record bytes read are 6 % of what it writes at 8 peers); and the
    library's data-movement reference kernels (spl_calib.h), which move each codec kernel's
    bytes the way that kernel does (bulk copies into a stage, its stores, its CTA shape) with
    none of its arithmetic.  Not a codec step."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    n = args.elements
    a = torch.rand(n, device=dev)
    b = torch.rand(n, device=dev)
    c = torch.empty(n, device=dev)
    d = torch.empty(n, device=dev)
    e = torch.empty(n, dtype=torch.int32, device=dev)
    kernels = {"copy (read 4 B, write 4 B per value)": (lambda: c.copy_(a), 8 * n),
               "add (read 8 B, write 4 B)": (lambda: torch.add(a, b, out=c), 12 * n),
               "frexp (read 4 B, write 8 B)": (lambda: torch.frexp(a, out=(c, e)), 12 * n),
               "fill (write 4 B)": (lambda: c.fill_(1.0), 4 * n)}
    if n % CHUNK == 0:
        for order, pers in (("codec order", False), ("one persistent wave", True)):
            kernels[f"the sender's movement (e and delta staged by bulk copies, plain stores), "
                    f"{order}"] = (lambda pers=pers: spl.calib_moves(
                        spl.CALIB_SENDER_MOVES, a, b, out0=c, persistent=pers), 12 * n)
            kernels[f"the receiver's movement (theta staged, mean and theta stored), "
                    f"{order}"] = (lambda pers=pers: spl.calib_moves(
                        spl.CALIB_RECEIVER_MOVES, a, out0=c, out1=d, persistent=pers), 12 * n)
    peak, kind = read_peaks()
    rows = {}
    for name, (fn, nbytes) in kernels.items():
        for _ in range(args.warmup):
            fn()
        times = []
        for _ in range(args.steps):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record()
            fn()
            s1.record()
            torch.cuda.synchronize(dev)
            times.append(s0.elapsed_time(s1) / 1e3)
        best = min(times)
        gbs = nbytes / best / 1e9
        rows[name] = {"ms": round(1e3 * best, 4), "GB/s": round(gbs, 1),
                      "frac_of_hbm": round(gbs / peak, 4),
                      "mean_ms": round(1e3 * sum(times) / len(times), 4)}
    line = {"metric": "HBM bandwidth of plain streaming kernels by read/write mix (context)",
            "value": rows["add (read 8 B, write 4 B)"]["GB/s"], "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"hbm-mix: torch copy_, add, frexp and fill_, and the codec "
                                   f"kernels' data movement alone, on {n} fp32 values",
                       "peak_gbs": peak, "peak_kind": kind, "kernels": rows}}
    print(json.dumps(line), flush=True)
    return 0


def run_sharded(args, dev, rank, world):
    """One peer's 2^30-value pseudo-gradient spread over the node's GPUs (chunk-sharded): each
    rank compresses its slice, the ranks all-gather the records (the peer's whole payload on
    every rank), and each rank decodes the 24 peers' records of its own chunk range into its
    slice of the mean fused with the outer step.  Total work is fixed as N grows (strong
    scaling); the value is the whole tensor's algorithmic bytes over the slowest rank's time."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl
    from compressed_pseudo_gradient_gb300 import sharded, synth

    n = args.elements
    C = (n + CHUNK - 1) // CHUNK
    lo, hi = sharded.shard_range(n, world, rank)
    m = hi - lo
    base = rank_seed_base(0)
    deltas = [synth.laplace(m, 1e-4, synth.generator(sd + 7 * rank, dev), dev)
              for sd in round_seeds(base)]
    ef = torch.zeros(m, dtype=torch.float32, device=dev)
    pls, scs = [], []
    tmp = torch.empty(m, dtype=torch.float32, device=dev)
    for p in range(PEERS):   # the peers' records of this rank's chunk range
        d = synth.laplace(m, 1e-4, synth.generator(base + 1 + p + 1000 * rank, dev), dev)
        tmp.zero_()
        a, b = spl.ef_compress(d, tmp, BETA)
        pls.append(a)
        scs.append(b)
        del d
    del tmp
    theta = synth.theta(m, synth.generator(base + 5000 + rank, dev), dev)
    mean = torch.empty(m, dtype=torch.float32, device=dev)
    state = {"round": 0}

    def step(ev=None):
        if ev:
            ev[0].record()
        pl, sc = sharded.compress_shard(deltas[state["round"] % ROUNDS], ef, BETA)
        state["round"] += 1
        if ev:
            ev[1].record()
        full_pl, full_sc = sharded.gather_records(pl, sc, C)
        if ev:
            ev[2].record()
        sharded.decode_shard(pls, scs, n, mean=mean, theta=theta, lr=LR)
        if ev:
            ev[3].record()
        return full_pl

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(dev)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(smi_id(dev)) as clk:
        start.record()
        for k in range(args.steps):
            step(evs[k])
        end.record()
        torch.cuda.synchronize(dev)
    barrier(dev)
    t_max = max_over_ranks(start.elapsed_time(end) / 1e3, dev)
    if rank != 0:
        return 0
    step_bytes = compress_bytes(n, C) + decode_bytes(n, C, PEERS)
    ms = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(3)]
    peak, kind = read_peaks()
    value = step_bytes / (t_max / args.steps) / 1e9
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_max / args.steps, 4), "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"chunk-sharded: one {n}-value pseudo-gradient over {world} "
                                   f"GPU(s): compress of each slice, all-gather of the records, "
                                   f"decode of 24 peers' records of each rank's chunk range "
                                   f"fused with the outer step",
                       "n": n, "chunks": C, "peers": PEERS, "parallelism": f"chunk-sharded x{world}",
                       "rank0_slice": [lo, hi],
                       "rank0_ms": {"compress": round(ms[0], 4), "all_gather": round(ms[1], 4),
                                    "decode": round(ms[2], 4)},
                       "frac_of_hbm_per_gpu": round(value / world / peak, 4), "peak_kind": kind},
            "clocks": clk.summary(), "gpu_launches": 2 * args.steps}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, dev, rank, world):
    import torch

    buf = setup_workload(dev, seed_base=rank_seed_base(rank), n=args.elements)
    if args.decode_stats:
        import compressed_pseudo_gradient_gb300 as spl
        buf["stats"] = spl.new_peer_stats(PEERS, dev)
    for _ in range(args.warmup):
        gpu_step(buf)
    torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    launches = 0
    barrier(dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_id(dev)) as clk:
        start.record()
        for k in range(args.steps):
            launches += gpu_step(buf, evs[k])
        end.record()
        torch.cuda.synchronize(dev)
    barrier(dev)
    t_total = start.elapsed_time(end) / 1e3
    t_max = max_over_ranks(t_total, dev)
    comp_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    flags = int(buf["flags"].item())

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, buf, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_from_device(buf, args.cpu_chunks)
    return {"t_total": t_total, "t_max": t_max, "comp_ms": comp_ms, "dec_ms": dec_ms,
            "launches": launches, "clocks": clk.summary(), "flags": flags, "e2e": e2e,
            "cpu": cpu}


def run_e2e(args, buf, dev):
    """The same step through the public API with host buffers: H2D of the step's inputs
    (delta and the 24 peers' records and scales) from pinned memory, the two calls, and D2H
    of the step's result (this peer's records and scales).  Two sets of device inputs: step
    i + 1's copies run on a copy stream while step i computes (each step still copies all of
    its inputs and reads back its result inside the timed region).  One pinned host delta
    serves every step: the copy's cost does not depend on its contents."""
    import torch
    import compressed_pseudo_gradient_gb300 as spl

    h_delta = buf["delta"].cpu().pin_memory()
    h_pl = [p.cpu().pin_memory() for p in buf["peers_pl"]]
    h_sc = [s.cpu().pin_memory() for s in buf["peers_sc"]]
    out_pl = torch.empty_like(buf["payload"], device="cpu").pin_memory()
    out_sc = torch.empty_like(buf["scales"], device="cpu").pin_memory()
    sets = [(torch.empty_like(buf["delta"]), [torch.empty_like(p) for p in buf["peers_pl"]],
             [torch.empty_like(s) for s in buf["peers_sc"]]) for _ in range(2)]
    h2d = h_delta.numel() * 4 + sum(p.numel() for p in h_pl) + sum(s.numel() * 4 for s in h_sc)
    d2h = out_pl.numel() + out_sc.numel() * 4
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(i):
        k = i % 2
        d_delta, d_pl, d_sc = sets[k]
        with torch.cuda.stream(copy):
            copy.wait_event(freed[k])          # step i - 2 has finished with this set
            d_delta.copy_(h_delta, non_blocking=True)
            for d, h in zip(d_pl, h_pl):
                d.copy_(h, non_blocking=True)
            for d, h in zip(d_sc, h_sc):
                d.copy_(h, non_blocking=True)
            copied[k].record(copy)

    def compute(i):
        k = i % 2
        d_delta, d_pl, d_sc = sets[k]
        comp.wait_event(copied[k])
        spl.ef_compress(d_delta, buf["ef"], BETA, payload=buf["payload"], scales=buf["scales"])
        spl.decode_aggregate(d_pl, d_sc, buf["n"], mean=buf["mean"], theta=buf["theta"], lr=LR)
        freed[k].record(comp)
        out_pl.copy_(buf["payload"], non_blocking=True)
        out_sc.copy_(buf["scales"], non_blocking=True)

    def run(steps, start=None):
        for e in freed:
            e.record(comp)
        if start is not None:
            copy.wait_stream(comp)             # no copy starts before the start event
        issue_copy(0)
        for i in range(steps):
            if i + 1 < steps:
                issue_copy(i + 1)
            compute(i)

    run(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    steps = max(1, args.e2e_steps)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dev)
    torch.cuda.synchronize(dev)
    start.record(comp)
    run(steps, start)
    end.record(comp)                           # after the last step's compute and D2H
    torch.cuda.synchronize(dev)
    barrier(dev)
    t = max_over_ranks(start.elapsed_time(end) / 1e3, dev)
    return {"seconds": t, "steps": steps, "h2d": h2d, "d2h": d2h}


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (the GPU arm's cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------------------------
def time_oracle(sample, threads: int):
    """Time the oracle over the sample's chunk ranges on `threads` host threads (ctypes
    releases the GIL).  Returns seconds for one pass (compress + decode with outer step)."""
    import numpy as np
    import oracle

    S = sample["chunks"]
    bounds = np.linspace(0, S, threads + 1).astype(int)

    def work(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi <= lo:
            return
        a, b = lo * CHUNK, hi * CHUNK
        ef = sample["ef"][a:b].copy()
        oracle.ef_compress(sample["delta"][a:b], ef, BETA)
        th = sample["theta"][a:b].copy()
        oracle.decode_aggregate([p[lo:hi] for p in sample["peers_pl"]],
                                [s[lo:hi] for s in sample["peers_sc"]], b - a, theta=th, lr=LR)

    oracle.build()
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, range(threads)))
    return time.perf_counter() - t0


def cpu_sample_bytes(S: int) -> int:
    return compress_bytes(S * CHUNK, S) + decode_bytes(S * CHUNK, S, PEERS)


def cpu_baseline_from_device(buf, chunks: int):
    """The oracle on the first `chunks` chunks of the same workload (copied from the GPU)."""
    S = min(chunks, (buf["n"] + CHUNK - 1) // CHUNK)
    sample = {
        "chunks": S,
        "delta": buf["delta"][:S * CHUNK].cpu().numpy(),
        "ef": buf["ef"][:S * CHUNK].cpu().numpy(),
        "theta": buf["theta"][:S * CHUNK].cpu().numpy(),
        "peers_pl": [p[:S].cpu().numpy() for p in buf["peers_pl"]],
        "peers_sc": [s[:S].cpu().numpy() for s in buf["peers_sc"]],
    }
    threads = os.cpu_count() or 1
    secs = time_oracle(sample, threads)
    # one core, on the first eighth of the sample (the same code on one thread)
    S1 = max(1, S // 8)
    one = {k: (v[:S1 * CHUNK] if k in ("delta", "ef", "theta") else v) for k, v in sample.items()}
    one["chunks"] = S1
    one["peers_pl"] = [p[:S1] for p in sample["peers_pl"]]
    one["peers_sc"] = [s[:S1] for s in sample["peers_sc"]]
    secs1 = time_oracle(one, 1)
    return {"value": round(cpu_sample_bytes(S) / secs / 1e9, 4), "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": f"first {S} of {N_CHUNKS} chunks of the same workload (compress + "
                      f"24-peer decode with outer step), one pass, {secs:.2f} s wall on "
                      f"{threads} host threads",
            "single_core": {"value": round(cpu_sample_bytes(S1) / secs1 / 1e9, 4),
                            "unit": "GB/s", "cores": 1,
                            "sample": f"first {S1} chunks, one pass, {secs1:.2f} s on one "
                                      f"host thread"}}


def make_cpu_sample(S: int, seed_base: int = 1):
    """Host-generated sample of the workload for the reference arm (same recipe)."""
    import numpy as np
    import torch
    import oracle
    from compressed_pseudo_gradient_gb300 import synth

    n = S * CHUNK
    cpu = torch.device("cpu")
    delta = synth.laplace(n, 1e-4, synth.generator(seed_base, cpu), cpu).numpy()
    peer_deltas = [synth.laplace(n, 1e-4, synth.generator(seed_base + 1 + p, cpu), cpu).numpy()
                   for p in range(PEERS)]

    def peer(d):   # the oracle's C calls release the GIL: the peers compress in parallel
        pl, sc, _ = oracle.ef_compress(d, np.zeros(n, np.float32), BETA)
        return pl, sc
    with ThreadPoolExecutor(max_workers=min(PEERS, os.cpu_count() or 1)) as ex:
        out = list(ex.map(peer, peer_deltas))
    pls = [o[0] for o in out]
    scs = [o[1] for o in out]
    theta = synth.theta(n, synth.generator(seed_base + 5000, cpu), cpu).numpy()
    return {"chunks": S, "delta": delta, "ef": np.zeros(n, np.float32), "theta": theta,
            "peers_pl": pls, "peers_sc": scs}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    S = args.cpu_chunks
    sample = make_cpu_sample(S)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        time_oracle(sample, threads)
    secs = [time_oracle(sample, threads) for _ in range(args.steps)]
    total = sum(secs)
    value = cpu_sample_bytes(S) * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n": N_ELEMS, "chunks": N_CHUNKS, "peers": PEERS,
                   "step_sample_chunks": S},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{S} chunks of the workload per step (compress + 24-peer "
                                   f"decode with outer step), host-generated with the same "
                                   f"recipe"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-chunks", type=int, default=32768)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the heavy-tailed bf16 and decoder-layer sub-records")
    ap.add_argument("--workload", default="receive",
                    choices=["receive", "heavy_tail_bf16", "decoder_layer", "tiny", "offload",
                             "codecs", "sharded", "hbm-mix"],
                    help="receive (default): the headline step; the others time one round of "
                         "another workload on one GPU")
    ap.add_argument("--decode-stats", action="store_true",
                    help="also gather the per-peer statistics in the receive pass")
    ap.add_argument("--elements", type=int, default=N_ELEMS,
                    help="pseudo-gradient size; smaller than 2^30 only for profiling captures")
    ap.add_argument("--layer-scale", type=int, default=1,
                    help="decoder_layer only: divide every tensor's rows by this (a profiling "
                         "case of the same shapes' row width and data)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        return run_reference(args)

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the default arm")
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.workload == "hbm-mix":
        return run_hbm_mix(args, dev)
    if args.workload == "sharded":
        dist_init("nccl")
        return run_sharded(args, dev, rank, world)
    if args.workload != "receive":
        if world != 1:
            raise SystemExit("--workload other than receive and sharded runs on one GPU")
        if args.workload == "offload":
            return run_offload(args, dev)
        if args.workload == "codecs":
            return run_codecs(args, dev)
        return run_other_workload(args, dev)
    dist_init("nccl")
    r = run_gpu(args, dev, rank, world)
    if rank != 0:
        return 0
    others = None
    movement = None
    n = args.elements
    C = (n + CHUNK - 1) // CHUNK
    if world == 1 and not args.no_other_workloads and args.elements == N_ELEMS:
        # the other two single-GPU workloads and the kernels' own data movement, timed after
        # the headline step (their own buffers; the headline's are released first)
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        steps = max(args.steps, 20)
        movement = movement_record(dev, n, C, steps, args.warmup,
                                   statistics.mean(r["comp_ms"]), statistics.mean(r["dec_ms"]))
        others = [other_workload_record(name, dev, steps, args.warmup)
                  for name in ("heavy_tail_bf16", "decoder_layer")]

    step_bytes = compress_bytes(n, C) + decode_bytes(n, C, PEERS)
    comp_avg = statistics.mean(r["comp_ms"]) / 1e3
    dec_avg = statistics.mean(r["dec_ms"]) / 1e3
    comp_gbs = compress_bytes(n, C) / comp_avg / 1e9
    dec_gbs = decode_bytes(n, C, PEERS) / dec_avg / 1e9
    peak, peak_kind = read_peaks()
    dominant = "ef_compress" if sum(r["comp_ms"]) >= sum(r["dec_ms"]) else "decode_aggregate"
    achieved = comp_gbs if dominant == "ef_compress" else dec_gbs
    value = aggregate_value(step_bytes, world, r["t_max"] / args.steps)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * r["t_max"] / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": WORKLOAD if n == N_ELEMS else f"profiling case: {n} values, same recipe",
            "n": n, "chunks": C, "peers": PEERS, "beta": BETA, "lr": LR, "rounds": ROUNDS,
            "step_bytes": step_bytes,
            "l2": "inputs (4 GiB per dense array) far exceed L2; no flush",
            "parallelism": f"independent peer per GPU x{world}",
            "ef_compress": {"ms": round(1e3 * comp_avg, 4), "GB/s": round(comp_gbs, 1),
                            "frac_of_hbm": round(comp_gbs / peak, 4),
                            "Gelem/s": round(n / comp_avg / 1e9, 2)},
            "decode_aggregate": {"ms": round(1e3 * dec_avg, 4), "GB/s": round(dec_gbs, 1),
                                 "frac_of_hbm": round(dec_gbs / peak, 4),
                                 "Gelem/s": round(n / dec_avg / 1e9, 2)},
            "device_flags": r["flags"],
            "decode_stats": bool(args.decode_stats),
        },
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": committed_traffic(dominant)},
        "clocks": r["clocks"],
        "gpu_launches": r["launches"],
    }
    if r["e2e"] is not None:
        e = r["e2e"]
        line["e2e"] = {"value": round(aggregate_value(step_bytes, world, e["seconds"] / e["steps"]), 2),
                       "unit": "GB/s", "h2d_bytes_per_step": e["h2d"],
                       "d2h_bytes_per_step": e["d2h"], "steps": e["steps"]}
    if r["cpu"] is not None:
        line["cpu_baseline"] = r["cpu"]
    if movement is not None:
        line["config"]["data_movement"] = movement
    if others is not None:
        line["config"]["other_workloads"] = others
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
